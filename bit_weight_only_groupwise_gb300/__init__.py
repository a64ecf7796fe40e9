"""Groupwise int4/int5/FP8 weight-only dequant-GEMM for GB300 (sm_103a).

Python binding of the C-ABI library ``_lib/libqgemm.so`` (declared in
``include/qgemm.h``).  Every function here has the name of the C entry point
it calls and does argument marshalling only: device pointers and streams are
taken from torch tensors and streams (or passed as plain integers), and the
status code is returned as the C function returns it.  All computation runs
in the library's CUDA kernels; there is no fallback: if the library is
missing the first call raises.

``GroupwiseWeights`` is a convenience holder that allocates the packed
buffer and the workspace with torch and binds them to a plan.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libqgemm.so")

QGEMM_OK = 0
QGEMM_ERR_INVALID_ARG = 1
QGEMM_ERR_SHAPE = 2
QGEMM_ERR_ALIGNMENT = 3
QGEMM_ERR_T_OUT_OF_DOMAIN = 4
QGEMM_ERR_WORKSPACE = 5
QGEMM_ERR_CUDA = 6
QGEMM_ERR_TIMEOUT = 7
QGEMM_ERR_UNSUPPORTED = 8

QGEMM_INT4 = 4
QGEMM_INT5 = 5
QGEMM_FP8 = 8
QGEMM_NVFP4 = 16

QGEMM_EPILOGUE_STORE = 0
QGEMM_EPILOGUE_ADD = 1
QGEMM_EPILOGUE_SWIGLU = 2
QGEMM_OUT_F32 = 0
QGEMM_OUT_BF16 = 1

# every symbol include/qgemm.h declares
EXPORTS = [
    "qgemm_status_string", "qgemm_packed_bytes", "qgemm_pack_weights", "qgemm_plan",
    "qgemm_plan_workspace_bytes", "qgemm_plan_bind", "qgemm_run", "qgemm_run_multi",
    "qgemm_plan_destroy", "qgemm_plan_route", "qgemm_route_name", "qgemm_launch_count",
    "qgemm_device_status", "qgemm_plan_set_pdl", "qgemm_pair_packed_bytes", "qgemm_pack_pair",
    "qgemm_plan_set_epilogue", "qgemm_run_ex", "qgemm_selftest_timeout", "qgemm_plan_force_route",
    "qgemm_run_noalloc", "qgemm_plan_set_tensor_scale",
]

_lock = threading.Lock()
_lib = None


class QgemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {qgemm_status_string(status)} ({status})" if what else qgemm_status_string(status))


def _declare(lib):
    c = ctypes
    vp, i32, sz, u64 = c.c_void_p, c.c_int, c.c_size_t, c.c_uint64
    sig = {
        "qgemm_status_string": ([i32], c.c_char_p),
        "qgemm_packed_bytes": ([i32, i32, i32], sz),
        "qgemm_pack_weights": ([i32, i32, i32, vp, vp, vp, vp], i32),
        "qgemm_plan": ([i32, i32, i32, i32, c.POINTER(vp)], i32),
        "qgemm_plan_workspace_bytes": ([vp], sz),
        "qgemm_plan_bind": ([vp, vp, vp, sz], i32),
        "qgemm_run": ([vp, vp, i32, vp, vp], i32),
        "qgemm_run_multi": ([c.POINTER(vp), i32, vp, i32, c.POINTER(vp), vp], i32),
        "qgemm_plan_destroy": ([vp], i32),
        "qgemm_plan_route": ([vp, i32], i32),
        "qgemm_route_name": ([i32], c.c_char_p),
        "qgemm_launch_count": ([], u64),
        "qgemm_device_status": ([vp, i32], i32),
        "qgemm_plan_set_pdl": ([vp, i32], i32),
        "qgemm_pair_packed_bytes": ([i32, i32, i32], sz),
        "qgemm_pack_pair": ([i32, i32, i32, vp, vp, vp, vp, vp, vp], i32),
        "qgemm_plan_set_epilogue": ([vp, i32, i32], i32),
        "qgemm_run_ex": ([vp, vp, i32, vp, vp, vp], i32),
        "qgemm_selftest_timeout": ([vp], i32),
        "qgemm_plan_force_route": ([vp, i32], i32),
        "qgemm_run_noalloc": ([vp, vp, vp, i32, vp, vp], i32),
        "qgemm_plan_set_tensor_scale": ([vp, c.c_float], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def load(path: str | None = None):
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"qgemm CUDA library not found at {p}; build it with "
                    "`python -m bit_weight_only_groupwise_gb300.build` (no CPU fallback exists)")
            lib = _declare(ctypes.CDLL(p))
            if path is not None:
                return lib
            _lib = lib
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


# ------------------------------------------------------------ C entry points

def qgemm_status_string(status: int) -> str:
    return load().qgemm_status_string(status).decode()


def qgemm_packed_bytes(N: int, K: int, codec: int) -> int:
    return load().qgemm_packed_bytes(N, K, codec)


def qgemm_pack_weights(codec, N, K, codes_canonical_dev, scales_fp16_dev, packed_dev, stream=None) -> int:
    return load().qgemm_pack_weights(codec, N, K, _ptr(codes_canonical_dev), _ptr(scales_fp16_dev),
                                     _ptr(packed_dev), _stream(stream))


def qgemm_plan(N: int, K: int, codec: int, T_max: int):
    """(status, plan handle)."""
    h = ctypes.c_void_p()
    st = load().qgemm_plan(N, K, codec, T_max, ctypes.byref(h))
    return st, h.value


def qgemm_plan_workspace_bytes(plan) -> int:
    return load().qgemm_plan_workspace_bytes(plan)


def qgemm_plan_bind(plan, packed_dev, workspace_dev, ws_bytes: int) -> int:
    return load().qgemm_plan_bind(plan, _ptr(packed_dev), _ptr(workspace_dev), ws_bytes)


def qgemm_run(plan, X, T: int, Y, stream=None) -> int:
    return load().qgemm_run(plan, _ptr(X), T, _ptr(Y), _stream(stream))


def qgemm_run_multi(plans, X, T: int, Ys, stream=None) -> int:
    n = len(plans)
    parr = (ctypes.c_void_p * max(n, 1))(*plans)
    yarr = (ctypes.c_void_p * max(len(Ys), 1))(*[_ptr(y) for y in Ys])
    return load().qgemm_run_multi(parr, n, _ptr(X), T, yarr, _stream(stream))


def qgemm_run_noalloc(plan, packed_dev, X, T: int, Y, stream=None) -> int:
    """qgemm_run on the tcgen05 route with the library's own scratch array, for
    callers that cannot allocate device memory (see include/qgemm.h)."""
    return load().qgemm_run_noalloc(plan, _ptr(packed_dev), _ptr(X), T, _ptr(Y), _stream(stream))


def qgemm_plan_destroy(plan) -> int:
    return load().qgemm_plan_destroy(plan)


def qgemm_pair_packed_bytes(F: int, K: int, codec: int) -> int:
    return load().qgemm_pair_packed_bytes(F, K, codec)


def qgemm_pack_pair(codec, F, K, gate_codes_dev, gate_scales_dev, up_codes_dev, up_scales_dev, packed_dev,
                    stream=None) -> int:
    return load().qgemm_pack_pair(codec, F, K, _ptr(gate_codes_dev), _ptr(gate_scales_dev), _ptr(up_codes_dev),
                                  _ptr(up_scales_dev), _ptr(packed_dev), _stream(stream))


def qgemm_plan_set_epilogue(plan, epilogue: int, out: int = QGEMM_OUT_F32) -> int:
    return load().qgemm_plan_set_epilogue(plan, epilogue, out)


def qgemm_run_ex(plan, X, T: int, R, Y, stream=None) -> int:
    return load().qgemm_run_ex(plan, _ptr(X), T, _ptr(R), _ptr(Y), _stream(stream))


def qgemm_plan_set_tensor_scale(plan, scale: float) -> int:
    return load().qgemm_plan_set_tensor_scale(plan, float(scale))


def qgemm_plan_set_pdl(plan, enable: bool) -> int:
    return load().qgemm_plan_set_pdl(plan, 1 if enable else 0)


def qgemm_plan_route(plan, T: int) -> int:
    return load().qgemm_plan_route(plan, T)


def qgemm_plan_force_route(plan, route: int) -> int:
    return load().qgemm_plan_force_route(plan, route)


def qgemm_route_name(route: int) -> str:
    return load().qgemm_route_name(route).decode()


def qgemm_launch_count() -> int:
    return load().qgemm_launch_count()


def qgemm_selftest_timeout(stream=None) -> int:
    return load().qgemm_selftest_timeout(_stream(stream))


def qgemm_device_status(stream=None, clear: bool = False) -> int:
    return load().qgemm_device_status(_stream(stream), 1 if clear else 0)


def check(status: int, what: str = "") -> None:
    if status != QGEMM_OK:
        raise QgemmError(status, what)


# ------------------------------------------------------------ convenience holders

def _check_tensor(t, shape, dtypes, device, what):
    """Raise QgemmError(QGEMM_ERR_SHAPE) unless t is a contiguous tensor of
    the given shape and one of the given dtypes on the given device.  The C
    entry points see only pointers, so a wrong extent here would make a
    kernel read or write past a buffer."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise QgemmError(QGEMM_ERR_INVALID_ARG, f"{what}: expected a torch tensor, got {type(t).__name__}")
    if t.dtype not in dtypes:
        raise QgemmError(QGEMM_ERR_SHAPE, f"{what}: dtype {t.dtype}, expected one of {list(dtypes)}")
    if tuple(t.shape) != tuple(shape):
        raise QgemmError(QGEMM_ERR_SHAPE, f"{what}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise QgemmError(QGEMM_ERR_SHAPE, f"{what}: not contiguous")
    if t.device != device:
        raise QgemmError(QGEMM_ERR_INVALID_ARG, f"{what}: on {t.device}, expected {device}")


def _x_dtypes():
    import torch
    # bf16 values, or their bit patterns in a 16-bit integer tensor
    return (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)


def _check_x(X, K, device):
    import torch
    if not isinstance(X, torch.Tensor) or X.dim() != 2:
        raise QgemmError(QGEMM_ERR_SHAPE, "X: expected a 2-D tensor [T, K]")
    _check_tensor(X, (X.shape[0], K), _x_dtypes(), device, "X")
    return X.shape[0]


def _to_dev(a, dtype, dev):
    import numpy as np
    import torch
    if isinstance(a, np.ndarray):
        a = torch.from_numpy(np.ascontiguousarray(a).view(dtype))
    return a.to(dev).contiguous()


class GroupwiseWeights:
    """One packed weight matrix bound to a plan (device memory from torch).

    ``codes_canonical`` and ``scales_fp16`` are the canonical packed codes
    (uint8 [N, row_bytes]: K/2 bytes per row for int4, 5K/8 for int5, K for
    FP8) and fp16 bit patterns (uint16/int16 [N, K/64]), as numpy arrays or
    torch tensors on the host or the device.  ``epilogue`` and ``out`` select
    a fused output (residual add) and the output type (fp32 or bf16).
    """

    def __init__(self, codec: int, N: int, K: int, codes_canonical, scales_fp16, T_max: int,
                 device="cuda", stream=None, epilogue: int = QGEMM_EPILOGUE_STORE, out: int = QGEMM_OUT_F32,
                 tensor_scale: float | None = None):
        import numpy as np
        import torch
        self.codec, self.N, self.K, self.T_max = codec, N, K, T_max
        self.epilogue, self.out = epilogue, out
        dev = torch.device(device)
        if dev.type == "cuda" and dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self.tensor_scale = tensor_scale
        codes = _to_dev(codes_canonical, np.uint8, dev)
        # NVFP4: UE4M3 block-scale bytes [N, K/16]; otherwise fp16 patterns
        scales = _to_dev(scales_fp16, np.uint8 if codec == QGEMM_NVFP4 else np.int16, dev)
        nbytes = qgemm_packed_bytes(N, K, codec)
        if nbytes == 0:
            raise QgemmError(QGEMM_ERR_SHAPE, "qgemm_packed_bytes")
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        check(qgemm_pack_weights(codec, N, K, codes, scales, self.packed, stream), "qgemm_pack_weights")
        self._make_plan(dev)

    def _make_plan(self, dev):
        import torch
        st, self.plan = qgemm_plan(self.N, self.K, self.codec, self.T_max)
        check(st, "qgemm_plan")
        if (self.epilogue, self.out) != (QGEMM_EPILOGUE_STORE, QGEMM_OUT_F32):
            check(qgemm_plan_set_epilogue(self.plan, self.epilogue, self.out), "qgemm_plan_set_epilogue")
        if getattr(self, "tensor_scale", None) is not None:
            check(qgemm_plan_set_tensor_scale(self.plan, self.tensor_scale), "qgemm_plan_set_tensor_scale")
        wsb = qgemm_plan_workspace_bytes(self.plan)
        self.workspace = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)
        check(qgemm_plan_bind(self.plan, self.packed, self.workspace, self.workspace.numel()), "qgemm_plan_bind")

    def route(self, T: int) -> str:
        return qgemm_route_name(qgemm_plan_route(self.plan, T))

    def run(self, X, Y=None, stream=None, R=None):
        """Y = epilogue(X[T, K] (bf16) . deq(W)^T): fp32 or bf16 [T, N] ([T, F]
        for a SwiGLU pair); R is the fp32 [T, N] residual of an ADD plan.

        X, Y and R must be contiguous tensors of exactly these shapes and
        dtypes on the weights' device (X may hold bf16 bit patterns as int16);
        anything else raises QgemmError before any launch."""
        import torch
        T = _check_x(X, self.K, self.device)
        ydtype = torch.bfloat16 if self.out == QGEMM_OUT_BF16 else torch.float32
        if Y is None:
            Y = torch.empty((T, self.N), dtype=ydtype, device=X.device)
        else:
            _check_tensor(Y, (T, self.N), (ydtype,), self.device, "Y")
        if R is not None:
            _check_tensor(R, (T, self.N), (torch.float32,), self.device, "R")
        if (self.epilogue, self.out) == (QGEMM_EPILOGUE_STORE, QGEMM_OUT_F32) and R is None:
            check(qgemm_run(self.plan, X, T, Y, stream), "qgemm_run")
        else:
            check(qgemm_run_ex(self.plan, X, T, R, Y, stream), "qgemm_run_ex")
        return Y

    def close(self):
        if getattr(self, "plan", None):
            qgemm_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def run_multi(weights, X, Ys=None, stream=None):
    """Several GroupwiseWeights (same K) over one shared X in one launch.

    X and every Ys[i] are checked as in GroupwiseWeights.run (X [T, K]
    bf16, Ys[i] fp32 [T, N_i], contiguous, on the weights' device)."""
    import torch
    if not weights:
        raise QgemmError(QGEMM_ERR_INVALID_ARG, "run_multi: no weights")
    dev = weights[0].device
    for w in weights:
        if w.K != weights[0].K:
            raise QgemmError(QGEMM_ERR_SHAPE, "run_multi: parents differ in K")
        if w.device != dev:
            raise QgemmError(QGEMM_ERR_INVALID_ARG, "run_multi: parents on different devices")
    T = _check_x(X, weights[0].K, dev)
    if Ys is None:
        Ys = [torch.empty((T, w.N), dtype=torch.float32, device=X.device) for w in weights]
    else:
        if len(Ys) != len(weights):
            raise QgemmError(QGEMM_ERR_INVALID_ARG, "run_multi: one output per parent")
        for i, (w, y) in enumerate(zip(weights, Ys)):
            _check_tensor(y, (T, w.N), (torch.float32,), dev, f"Ys[{i}]")
    check(qgemm_run_multi([w.plan for w in weights], X, T, Ys, stream), "qgemm_run_multi")
    return Ys


class SwiGLUPair(GroupwiseWeights):
    """The gate and up matrices of an MLP (F x K each, same codec) packed as one
    pair; ``run(X)`` returns silu(X . G^T) * (X . U^T), [T, F]."""

    def __init__(self, codec: int, F: int, K: int, gate_codes, gate_scales, up_codes, up_scales, T_max: int,
                 device="cuda", stream=None, out: int = QGEMM_OUT_F32, tensor_scale: float | None = None):
        import numpy as np
        import torch
        self.codec, self.N, self.K, self.T_max = codec, F, K, T_max
        self.epilogue, self.out = QGEMM_EPILOGUE_SWIGLU, out
        dev = torch.device(device)
        if dev.type == "cuda" and dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        nbytes = qgemm_pair_packed_bytes(F, K, codec)
        if nbytes == 0:
            raise QgemmError(QGEMM_ERR_SHAPE, "qgemm_pair_packed_bytes")
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.tensor_scale = tensor_scale
        sdt = np.uint8 if codec == QGEMM_NVFP4 else np.int16
        check(qgemm_pack_pair(codec, F, K, _to_dev(gate_codes, np.uint8, dev), _to_dev(gate_scales, sdt, dev),
                              _to_dev(up_codes, np.uint8, dev), _to_dev(up_scales, sdt, dev), self.packed,
                              stream), "qgemm_pack_pair")
        self._make_plan(dev)
