"""CPU oracle for the groupwise int4/int5 dequant-GEMM (Python loader).

TEST INFRASTRUCTURE: only the tests, the package entry point's smoke check
and the benchmark's CPU-baseline leg may import this module.  The product
path (the CUDA library and its binding) never imports or calls it.

``qgemm_oracle.c`` holds the arithmetic (plain fp64, single-threaded, the
definition written out); this file compiles it with gcc on first use and
marshals numpy arrays across ctypes.  Nothing here computes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qgemm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libqgemm_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c99", "-Wall", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into a shared library (gcc); returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    i32, ptr = ctypes.c_int, ctypes.c_void_p
    lib.qgemm_oracle_row_bytes.argtypes = [i32, i32]
    lib.qgemm_oracle_row_bytes.restype = i32
    lib.qgemm_oracle_groups.argtypes = [i32]
    lib.qgemm_oracle_groups.restype = i32
    lib.qgemm_oracle_unpack.argtypes = [i32, i32, i32, ptr, ptr]
    lib.qgemm_oracle_unpack.restype = i32
    lib.qgemm_oracle_dequant.argtypes = [i32, i32, i32, ptr, ptr, ptr]
    lib.qgemm_oracle_dequant.restype = i32
    lib.qgemm_oracle_gemm.argtypes = [i32, i32, i32, i32, ptr, ptr, ptr, ptr, ptr]
    lib.qgemm_oracle_gemm.restype = i32
    lib.qgemm_oracle_linear_add.argtypes = [i32, i32, i32, i32, ptr, ptr, ptr, ptr, ptr, ptr]
    lib.qgemm_oracle_linear_add.restype = i32
    lib.qgemm_oracle_swiglu.argtypes = [i32, ptr, ptr, ptr]
    lib.qgemm_oracle_swiglu.restype = i32
    lib.qgemm_oracle_nvfp4_blocks.argtypes = [i32]
    lib.qgemm_oracle_nvfp4_blocks.restype = i32
    lib.qgemm_oracle_dequant_nvfp4.argtypes = [i32, i32, ptr, ptr, ctypes.c_float, ptr]
    lib.qgemm_oracle_dequant_nvfp4.restype = i32
    lib.qgemm_oracle_gemm_nvfp4.argtypes = [i32, i32, i32, ptr, ptr, ctypes.c_float, ptr, ptr, ptr]
    lib.qgemm_oracle_gemm_nvfp4.restype = i32
    return lib


def load(path: str | None = None):
    """The compiled oracle (built on first use, rebuilt when the source is newer)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def row_bytes(bits: int, K: int) -> int:
    return load().qgemm_oracle_row_bytes(bits, K)


def unpack(bits: int, packed: np.ndarray, N: int, K: int, lib=None) -> np.ndarray:
    """int8 codes [N, K] read from the canonical packing."""
    lib = lib or load()
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros((N, K), np.int8)
    if lib.qgemm_oracle_unpack(bits, N, K, _p(packed), _p(out)) != 0:
        raise ValueError("oracle unpack: bad arguments")
    return out


def dequant(bits: int, packed: np.ndarray, scales: np.ndarray, N: int, K: int, lib=None) -> np.ndarray:
    """fp64 W[n, k] = s[n, k/64] * q[n, k]."""
    lib = lib or load()
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    out = np.zeros((N, K), np.float64)
    if lib.qgemm_oracle_dequant(bits, N, K, _p(packed), _p(scales), _p(out)) != 0:
        raise ValueError("oracle dequant: bad arguments")
    return out


def gemm(bits: int, packed: np.ndarray, scales: np.ndarray, x_bf16: np.ndarray,
         N: int, K: int, lib=None):
    """(Y, A): fp64 [T, N] result and sum of |products| for the tolerance."""
    lib = lib or load()
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T = x.shape[0]
    assert x.shape == (T, K), (x.shape, T, K)
    Y = np.zeros((T, N), np.float64)
    A = np.zeros((T, N), np.float64)
    if lib.qgemm_oracle_gemm(bits, N, K, T, _p(packed), _p(scales), _p(x), _p(Y), _p(A)) != 0:
        raise ValueError("oracle gemm: bad arguments")
    return Y, A


NVFP4 = 16   # codec id of NVFP4 weights (E2M1 codes, UE4M3 scale per 16 columns, fp32 tensor scale)


def dequant_nvfp4(codes_packed: np.ndarray, bscales: np.ndarray, tscale: float, N: int, K: int,
                  lib=None) -> np.ndarray:
    """fp64 W[n, k] = e2m1(c[n, k]) * ue4m3(b[n, k/16]) * tscale."""
    lib = lib or load()
    codes_packed = np.ascontiguousarray(codes_packed, dtype=np.uint8)
    bscales = np.ascontiguousarray(bscales, dtype=np.uint8)
    out = np.zeros((N, K), np.float64)
    if lib.qgemm_oracle_dequant_nvfp4(N, K, _p(codes_packed), _p(bscales), float(tscale), _p(out)) != 0:
        raise ValueError("oracle dequant_nvfp4: bad arguments")
    return out


def gemm_nvfp4(codes_packed: np.ndarray, bscales: np.ndarray, tscale: float, x_bf16: np.ndarray, N: int, K: int,
               lib=None):
    """(Y, A) of an NVFP4 matrix, as gemm() for the other codecs."""
    lib = lib or load()
    codes_packed = np.ascontiguousarray(codes_packed, dtype=np.uint8)
    bscales = np.ascontiguousarray(bscales, dtype=np.uint8)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T = x.shape[0]
    assert x.shape == (T, K), (x.shape, T, K)
    Y = np.zeros((T, N), np.float64)
    A = np.zeros((T, N), np.float64)
    if lib.qgemm_oracle_gemm_nvfp4(N, K, T, _p(codes_packed), _p(bscales), float(tscale), _p(x), _p(Y),
                                   _p(A)) != 0:
        raise ValueError("oracle gemm_nvfp4: bad arguments")
    return Y, A


def gemm_parent(parent: dict, x_bf16: np.ndarray, lib=None):
    """Oracle on one weight matrix as drawn by the input generator."""
    if parent["bits"] == NVFP4:
        return gemm_nvfp4(parent["packed"], parent["scales"], parent["tscale"], x_bf16, parent["N"], parent["K"],
                          lib=lib)
    return gemm(parent["bits"], parent["packed"], parent["scales"], x_bf16,
                parent["N"], parent["K"], lib=lib)


def linear_add(bits: int, packed: np.ndarray, scales: np.ndarray, x_bf16: np.ndarray, R: np.ndarray,
               N: int, K: int, lib=None):
    """(Y, A) of Y = R + X . deq(W)^T; R fp32 [T, N]."""
    lib = lib or load()
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T = x.shape[0]
    R = np.ascontiguousarray(R, dtype=np.float32)
    assert x.shape == (T, K) and R.shape == (T, N), (x.shape, R.shape, T, N, K)
    Y = np.zeros((T, N), np.float64)
    A = np.zeros((T, N), np.float64)
    if lib.qgemm_oracle_linear_add(bits, N, K, T, _p(packed), _p(scales), _p(x), _p(R), _p(Y), _p(A)) != 0:
        raise ValueError("oracle linear_add: bad arguments")
    return Y, A


def swiglu(g: np.ndarray, u: np.ndarray, lib=None) -> np.ndarray:
    """silu(g) * u elementwise in fp64 (g, u same shape)."""
    lib = lib or load()
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    assert g.shape == u.shape
    out = np.zeros(g.shape, np.float64)
    if lib.qgemm_oracle_swiglu(g.size, _p(g), _p(u), _p(out)) != 0:
        raise ValueError("oracle swiglu: bad arguments")
    return out


def swiglu_pair(gate: dict, up: dict, x_bf16: np.ndarray, lib=None):
    """(out, g, u, A_g, A_u): the SwiGLU of a gate/up pair of weight matrices
    as drawn by the input generator, with the plain results and their sums of
    |products| (for the tolerance)."""
    g, Ag = gemm_parent(gate, x_bf16, lib=lib)
    u, Au = gemm_parent(up, x_bf16, lib=lib)
    return swiglu(g, u, lib=lib), g, u, Ag, Au
