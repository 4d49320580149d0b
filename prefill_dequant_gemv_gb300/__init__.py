"""Python binding of the GB300 quantized GEMV / GEMM library (``libqgemv.so``).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  PyTorch provides device memory and streams.  The functions carry
the C ABI's names (see ``include/qgemv.h``); ``PackedWeight`` and the lower-case
helpers wrap them for torch tensors.

The library must have been built (``prefill_dequant_gemv_gb300.build.build()``);
importing the binding without it raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemv.so")

FMT_MLX_AFFINE4_G64, FMT_MXFP4, FMT_NVFP4, FMT_Q6K = 1, 2, 3, 4
OUT_F32, OUT_BF16 = 0, 1
STATUS = {0: "QG_OK", 1: "QG_ERR_INVALID_ARG", 2: "QG_ERR_UNSUPPORTED", 3: "QG_ERR_MISALIGNED",
          4: "QG_ERR_WORKSPACE_TOO_SMALL", 5: "QG_ERR_CUDA", 6: "QG_ERR_TIMEOUT"}


class QGError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class qg_weight(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("reserved", ctypes.c_int32), ("n", ctypes.c_int64),
                ("k", ctypes.c_int64), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("aux", ctypes.c_void_p), ("tensor_scale", ctypes.c_float), ("reserved2", ctypes.c_float)]


_lib = None
_P, _I64, _I, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_SIGNATURES = {
    "qg_status_str": (ctypes.c_char_p, [_I]),
    "qg_packed_sizes": (_I, [_I, _I64, _I64, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "qg_pack_host": (_I, [_I, _I64, _I64, _P, _P, _P, _P, _P, _P]),
    "qg_dequant": (_I, [ctypes.POINTER(qg_weight), _I, _P, _I64, _P]),
    "qg_gemv_workspace_size": (_SZ, [_I, _I64, _I64, _I]),
    "qg_workspace_init": (_I, [_P, _SZ, _P]),
    "qg_workspace_status": (_I, [_P, ctypes.POINTER(_I), _P]),
    "qgemv": (_I, [ctypes.POINTER(qg_weight), _P, _I, _I64, _P, _I64, _P, _I64, _P, _SZ, _P]),
    "qgemv_static_ws": (_I, [ctypes.POINTER(qg_weight), _P, _I, _I64, _P, _I64, _P, _I64, _P]),
    "qg_gemm_workspace_size": (_SZ, [_I, _I64, _I64, _I]),
    "qgemm": (_I, [ctypes.POINTER(qg_weight), _P, _I64, _I64, _P, _I64, _P, _I64, _P, _SZ, _P]),
}


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with prefill_dequant_gemv_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _check(st: int, what: str):
    if st != 0:
        raise QGError(st, what)


# ------------------------------------------------------------------ C ABI, same names
def qg_status_str(status: int) -> str:
    return lib().qg_status_str(status).decode()


def qg_packed_sizes(fmt: int, n: int, k: int):
    c, s, a = _SZ(), _SZ(), _SZ()
    _check(lib().qg_packed_sizes(fmt, n, k, ctypes.byref(c), ctypes.byref(s), ctypes.byref(a)), "qg_packed_sizes")
    return c.value, s.value, a.value


def qg_pack_host(fmt: int, n: int, k: int, codes: np.ndarray, scales: np.ndarray, aux: Optional[np.ndarray]):
    """Pack logical host arrays; returns (codes, scales, aux) uint8 numpy arrays (aux empty unless Q6_K)."""
    cb, sb, ab = qg_packed_sizes(fmt, n, k)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales)
    aux = None if aux is None else np.ascontiguousarray(aux)
    oc, os_, oa = np.empty(cb, np.uint8), np.empty(sb, np.uint8), np.empty(max(ab, 1), np.uint8)
    st = lib().qg_pack_host(fmt, n, k, codes.ctypes.data, scales.ctypes.data,
                            None if aux is None else aux.ctypes.data,
                            oc.ctypes.data, os_.ctypes.data, oa.ctypes.data if ab else None)
    _check(st, "qg_pack_host")
    return oc, os_, oa[:ab]


def qg_dequant(w: qg_weight, out_dtype: int, out_ptr: int, ldo: int, stream: int = 0):
    _check(lib().qg_dequant(ctypes.byref(w), out_dtype, out_ptr, ldo, stream), "qg_dequant")


def qg_gemv_workspace_size(fmt: int, n: int, k: int, m: int) -> int:
    return lib().qg_gemv_workspace_size(fmt, n, k, m)


def qg_workspace_init(ptr: int, nbytes: int, stream: int = 0):
    _check(lib().qg_workspace_init(ptr, nbytes, stream), "qg_workspace_init")


def qg_workspace_status(ptr: int, stream: int = 0) -> int:
    v = _I()
    _check(lib().qg_workspace_status(ptr, ctypes.byref(v), stream), "qg_workspace_status")
    return v.value


def qgemv(w: qg_weight, x_ptr: int, m: int, ldx: int, res_ptr: Optional[int], ldr: int, y_ptr: int, ldy: int,
          ws_ptr: int, ws_bytes: int, stream: int = 0):
    _check(lib().qgemv(ctypes.byref(w), x_ptr, m, ldx, res_ptr, ldr, y_ptr, ldy, ws_ptr, ws_bytes, stream),
           "qgemv")


def qg_gemm_workspace_size(fmt: int, n: int, k: int, m: int) -> int:
    return lib().qg_gemm_workspace_size(fmt, n, k, m)


def qgemm(w: qg_weight, x_ptr: int, m: int, ldx: int, res_ptr: Optional[int], ldr: int, y_ptr: int, ldy: int,
          ws_ptr: int, ws_bytes: int, stream: int = 0):
    _check(lib().qgemm(ctypes.byref(w), x_ptr, m, ldx, res_ptr, ldr, y_ptr, ldy, ws_ptr, ws_bytes, stream), "qgemm")


def qgemv_static_ws(w: qg_weight, x_ptr: int, m: int, ldx: int, res_ptr: Optional[int], ldr: int, y_ptr: int,
                    ldy: int, stream: int = 0):
    """qgemv without a workspace argument, for callers that cannot allocate device memory
    (its scratch is a fixed array inside the library, shared by all calls)."""
    _check(lib().qgemv_static_ws(ctypes.byref(w), x_ptr, m, ldx, res_ptr, ldr, y_ptr, ldy, stream), "qgemv_static_ws")


# ------------------------------------------------------------------ torch helpers
def _stream_ptr(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


class PackedWeight:
    """A packed weight resident in device memory plus its ``qg_weight`` descriptor."""

    def __init__(self, fmt: int, n: int, k: int, codes, scales, aux, tensor_scale: float = 1.0):
        self.fmt, self.n, self.k = fmt, n, k
        self.codes, self.scales, self.aux = codes, scales, aux  # torch uint8 device tensors
        self.tensor_scale = float(tensor_scale)
        self.desc = qg_weight(fmt, 0, n, k, codes.data_ptr(), scales.data_ptr(),
                              aux.data_ptr() if aux is not None else None, self.tensor_scale, 0.0)

    @property
    def nbytes(self) -> int:
        return self.codes.numel() + self.scales.numel() + (self.aux.numel() if self.aux is not None else 0)

    @staticmethod
    def from_logical(w, device="cuda") -> "PackedWeight":
        """Pack a logical weight (``workloads.QWeight``) on the host and copy it to ``device``."""
        import torch
        c, s, a = qg_pack_host(w.fmt, w.n, w.k, w.codes, w.scales, w.aux)
        tc = torch.from_numpy(c).to(device)
        ts_ = torch.from_numpy(s).to(device)
        ta = torch.from_numpy(a).to(device) if a.size else None
        return PackedWeight(w.fmt, w.n, w.k, tc, ts_, ta, w.tensor_scale if w.fmt == FMT_NVFP4 else 1.0)


class Workspace:
    """A zero-initialised device workspace (caller-owned memory for the kernels' split-K state)."""

    def __init__(self, nbytes: int, device="cuda"):
        import torch
        self.nbytes = max(int(nbytes), 256)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def status(self) -> int:
        return qg_workspace_status(self.ptr, _stream_ptr())


def dequant(pw: PackedWeight, out_dtype: int = OUT_F32):
    import torch
    dt = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
    ldo = (pw.k + 7) // 8 * 8
    out = torch.empty((pw.n, ldo), dtype=dt, device=pw.codes.device)
    qg_dequant(pw.desc, out_dtype, out.data_ptr(), ldo, _stream_ptr())
    return out[:, :pw.k]


def gemv(pw: PackedWeight, x, residual=None, out=None, workspace: Optional[Workspace] = None):
    """y = bf16(W x (+ residual)) for x bf16 [m, k] on the device, m = 1..4."""
    import torch
    m = x.shape[0]
    if out is None:
        out = torch.empty((m, (pw.n + 7) // 8 * 8), dtype=torch.bfloat16, device=x.device)[:, :pw.n]
    if workspace is None:
        workspace = Workspace(qg_gemv_workspace_size(pw.fmt, pw.n, pw.k, m), x.device)
    qgemv(pw.desc, x.data_ptr(), m, x.stride(0), None if residual is None else residual.data_ptr(),
          0 if residual is None else residual.stride(0), out.data_ptr(), out.stride(0), workspace.ptr,
          workspace.nbytes, _stream_ptr())
    return out


def gemm(pw: PackedWeight, x, residual=None, out=None, workspace: Optional[Workspace] = None):
    """y = bf16(W x (+ residual)) for x bf16 [m, k] on the device, any m (tokens)."""
    import torch
    m = x.shape[0]
    if out is None:
        out = torch.empty((m, (pw.n + 7) // 8 * 8), dtype=torch.bfloat16, device=x.device)[:, :pw.n]
    if workspace is None:
        workspace = Workspace(qg_gemm_workspace_size(pw.fmt, pw.n, pw.k, min(m, 2 ** 31 - 1)), x.device)
    qgemm(pw.desc, x.data_ptr(), m, x.stride(0), None if residual is None else residual.data_ptr(),
          0 if residual is None else residual.stride(0), out.data_ptr(), out.stride(0), workspace.ptr,
          workspace.nbytes, _stream_ptr())
    return out
