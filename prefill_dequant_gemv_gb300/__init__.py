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

FMT_MLX_AFFINE4_G64, FMT_MXFP4, FMT_NVFP4, FMT_Q6K, FMT_Q5_0, FMT_Q5_1, FMT_Q5_K = 1, 2, 3, 4, 5, 6, 7
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


class qg_moe_layer(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("hidden", ctypes.c_int64),
                ("ffn", ctypes.c_int64), ("gu_codes", ctypes.c_void_p), ("gu_scales", ctypes.c_void_p),
                ("gu_aux", ctypes.c_void_p), ("dn_codes", ctypes.c_void_p), ("dn_scales", ctypes.c_void_p),
                ("dn_aux", ctypes.c_void_p), ("tensor_scale", ctypes.c_float), ("has_shared", ctypes.c_int32),
                ("shared_gate_up", qg_weight), ("shared_down", qg_weight)]


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
    "qgemv_static_ws_status": (_I, [ctypes.POINTER(_I), _P]),
    "qg_gemm_workspace_size": (_SZ, [_I, _I64, _I64, _I]),
    "qgemm": (_I, [ctypes.POINTER(qg_weight), _P, _I64, _I64, _P, _I64, _P, _I64, _P, _SZ, _P]),
    "qmoe_route_workspace_size": (_SZ, [_I64, _I, _I]),
    "qmoe_route": (_I, [_P, _I64, _I, _I, _P, _P, _P, _SZ, _P]),
    "qmoe_workspace_size": (_SZ, [ctypes.POINTER(qg_moe_layer), _I64, _I]),
    "qmoe_ffn": (_I, [ctypes.POINTER(qg_moe_layer), _P, _I64, _I64, _I, _P, _P, _P, _P, _I64, _P, _SZ, _P]),
    "qgemm_grouped_workspace_size": (_SZ, [ctypes.POINTER(qg_moe_layer), _I64, _I, _I]),
    "qmoe_forward": (_I, [ctypes.POINTER(qg_moe_layer), _P, _I64, _I64, _P, _I, _P, _P, _P, _P, _SZ, _P, _I64, _P, _SZ,
                          _P]),
    "qgemm_grouped": (_I, [ctypes.POINTER(qg_moe_layer), _I, _P, _I64, _I64, _I, _P, _P, _P, _P, _I64, _P, _SZ, _P]),
    "qg_selftest_wait_timeout": (_I, [_P, _SZ, _P]),
    "qg_quant_act_nvfp4": (_I, [_P, _I64, _I64, _I64, ctypes.c_float, _P, _I64, _P, _I64, _P, _I64, _P]),
    "qgemm_w4a4_workspace_size": (_SZ, [_I, _I64, _I64, _I64]),
    "qgemm_w4a4": (_I, [ctypes.POINTER(qg_weight), _P, _I64, _I64, ctypes.c_float, _P, _I64, _P, _I64, _P, _SZ,
                        _P]),
}

QG_MOE_GATE_UP_SWIGLU = 1
QG_MOE_DOWN_COMBINE = 2


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
    """Pack logical host arrays; returns (codes, scales, aux) uint8 numpy arrays (aux empty unless Q6_K or
    Q5_K)."""
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


def qg_quant_act_nvfp4(x_ptr: int, m: int, k: int, ldx: int, act_scale: float, codes_ptr: Optional[int], ldc: int,
                       scales_ptr: Optional[int], lds: int, xe_ptr: Optional[int], lde: int, stream: int = 0):
    _check(lib().qg_quant_act_nvfp4(x_ptr, m, k, ldx, act_scale, codes_ptr, ldc, scales_ptr, lds, xe_ptr, lde, stream),
           "qg_quant_act_nvfp4")


def qgemm_w4a4_workspace_size(fmt: int, n: int, k: int, m: int) -> int:
    return lib().qgemm_w4a4_workspace_size(fmt, n, k, m)


def qgemm_w4a4(w: qg_weight, x_ptr: int, m: int, ldx: int, act_scale: float, res_ptr: Optional[int], ldr: int,
               y_ptr: int, ldy: int, ws_ptr: int, ws_bytes: int, stream: int = 0):
    _check(lib().qgemm_w4a4(ctypes.byref(w), x_ptr, m, ldx, act_scale, res_ptr, ldr, y_ptr, ldy, ws_ptr, ws_bytes,
                            stream), "qgemm_w4a4")


def qmoe_route_workspace_size(t: int, n_experts: int, topk: int) -> int:
    return lib().qmoe_route_workspace_size(t, n_experts, topk)


def qmoe_route(logits_ptr: int, t: int, n_experts: int, topk: int, ids_ptr: int, w_ptr: int, ws_ptr: int,
               ws_bytes: int, stream: int = 0):
    _check(lib().qmoe_route(logits_ptr, t, n_experts, topk, ids_ptr, w_ptr, ws_ptr, ws_bytes, stream), "qmoe_route")


def qmoe_workspace_size(layer: qg_moe_layer, t: int, topk: int) -> int:
    return lib().qmoe_workspace_size(ctypes.byref(layer), t, topk)


def qmoe_ffn(layer: qg_moe_layer, x_ptr: int, t: int, ldx: int, topk: int, w_ptr: int, gate_ptr: Optional[int],
             route_ws_ptr: int, out_ptr: int, ldo: int, ws_ptr: int, ws_bytes: int, stream: int = 0):
    _check(lib().qmoe_ffn(ctypes.byref(layer), x_ptr, t, ldx, topk, w_ptr, gate_ptr, route_ws_ptr, out_ptr, ldo,
                          ws_ptr, ws_bytes, stream), "qmoe_ffn")


def qmoe_forward(layer: qg_moe_layer, x_ptr: int, t: int, ldx: int, logits_ptr: int, topk: int,
                 gate_ptr: Optional[int], ids_ptr: int, w_ptr: int, route_ws_ptr: int, route_ws_bytes: int, out_ptr: int,
                 ldo: int, ws_ptr: int, ws_bytes: int, stream: int = 0):
    _check(lib().qmoe_forward(ctypes.byref(layer), x_ptr, t, ldx, logits_ptr, topk, gate_ptr, ids_ptr, w_ptr,
                              route_ws_ptr, route_ws_bytes, out_ptr, ldo, ws_ptr, ws_bytes, stream), "qmoe_forward")


def qgemm_grouped_workspace_size(layer: qg_moe_layer, t: int, topk: int, stage: int) -> int:
    return lib().qgemm_grouped_workspace_size(ctypes.byref(layer), t, topk, stage)


def qgemm_grouped(layer: qg_moe_layer, stage: int, in_ptr: int, t: int, ldi: int, topk: int, w_ptr: Optional[int],
                  gate_ptr: Optional[int], route_ws_ptr: int, out_ptr: int, ldo: int, ws_ptr: int, ws_bytes: int,
                  stream: int = 0):
    _check(lib().qgemm_grouped(ctypes.byref(layer), stage, in_ptr, t, ldi, topk, w_ptr, gate_ptr, route_ws_ptr,
                               out_ptr, ldo, ws_ptr, ws_bytes, stream), "qgemm_grouped")


def qgemv_static_ws(w: qg_weight, x_ptr: int, m: int, ldx: int, res_ptr: Optional[int], ldr: int, y_ptr: int,
                    ldy: int, stream: int = 0):
    """qgemv without a workspace argument, for callers that cannot allocate device memory
    (its scratch is a fixed array inside the library, shared by all calls)."""
    _check(lib().qgemv_static_ws(ctypes.byref(w), x_ptr, m, ldx, res_ptr, ldr, y_ptr, ldy, stream), "qgemv_static_ws")


def qgemv_static_ws_status(stream: int = 0) -> int:
    """Read and clear the status word of qgemv_static_ws's array on the current device
    (synchronises `stream`): QG_OK, or QG_ERR_TIMEOUT after a bounded wait gave up."""
    v = _I(0)
    _check(lib().qgemv_static_ws_status(ctypes.byref(v), stream), "qgemv_static_ws_status")
    return v.value


def qg_selftest_wait_timeout(ws_ptr: int, ws_bytes: int, stream: int = 0):
    """Launch the bounded-wait self-test (its wait runs out after the library's limit and
    records QG_ERR_TIMEOUT in the workspace status word)."""
    _check(lib().qg_selftest_wait_timeout(ws_ptr, ws_bytes, stream), "qg_selftest_wait_timeout")


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


def quant_act_nvfp4(x, act_scale: float):
    """NVFP4-quantise bf16 activations x [m, k] on the device (W4A4).  Returns (codes uint8 [m, k/2], two
    E2M1 codes a byte, the even k in the low nibble; scales uint8 [m, k/16] E4M3; xe bf16 [m, k], the exact
    expansion E4M3(S) * E2M1(code) without act_scale)."""
    import torch
    m, k = x.shape
    dev = x.device
    codes = torch.empty((m, (k // 2 + 7) // 8 * 8), dtype=torch.uint8, device=dev)
    scales = torch.empty((m, k // 16), dtype=torch.uint8, device=dev)
    xe = torch.empty((m, (k + 7) // 8 * 8), dtype=torch.bfloat16, device=dev)
    qg_quant_act_nvfp4(x.data_ptr(), m, k, x.stride(0), act_scale, codes.data_ptr(), codes.stride(0),
                       scales.data_ptr(), scales.stride(0), xe.data_ptr(), xe.stride(0), _stream_ptr())
    return codes[:, :k // 2], scales, xe[:, :k]


def gemm_w4a4(pw: PackedWeight, x, act_scale: float, residual=None, out=None, workspace: Optional[Workspace] = None):
    """y = bf16(W xq (+ residual)) with xq the NVFP4 quantisation of x (bf16 [m, k]) at tensor scale act_scale."""
    import torch
    m = x.shape[0]
    if out is None:
        out = torch.empty((m, (pw.n + 7) // 8 * 8), dtype=torch.bfloat16, device=x.device)[:, :pw.n]
    if workspace is None:
        workspace = Workspace(qgemm_w4a4_workspace_size(pw.fmt, pw.n, pw.k, m), x.device)
    qgemm_w4a4(pw.desc, x.data_ptr(), m, x.stride(0), act_scale, None if residual is None else residual.data_ptr(),
               0 if residual is None else residual.stride(0), out.data_ptr(), out.stride(0), workspace.ptr,
               workspace.nbytes, _stream_ptr())
    return out


class PackedMoE:
    """A mixture-of-experts layer packed on the host and resident in device memory: the
    routed experts' packed matrices back to back, the shared expert separate."""

    def __init__(self, layer, device="cuda"):
        import torch
        self.fmt, self.n_experts, self.hidden, self.ffn = layer.fmt, layer.n_experts, layer.hidden, layer.ffn

        def pack_all(ws):
            parts = [qg_pack_host(w.fmt, w.n, w.k, w.codes, w.scales, w.aux) for w in ws]
            out = []
            for i in range(3):
                cat = np.concatenate([p[i] for p in parts]) if parts[0][i].size else np.zeros(0, np.uint8)
                out.append(torch.from_numpy(cat).to(device) if cat.size else None)
            return out

        self.gu = pack_all(layer.gate_up)
        self.dn = pack_all(layer.down)
        self.shared = None
        if layer.shared_gate_up is not None:
            self.shared = (PackedWeight.from_logical(layer.shared_gate_up, device),
                           PackedWeight.from_logical(layer.shared_down, device))
        ts = layer.gate_up[0].tensor_scale if layer.fmt == FMT_NVFP4 else 1.0
        empty = qg_weight(layer.fmt, 0, 0, 0, None, None, None, 1.0, 0.0)
        self.desc = qg_moe_layer(
            layer.fmt, layer.n_experts, layer.hidden, layer.ffn,
            self.gu[0].data_ptr(), self.gu[1].data_ptr(), self.gu[2].data_ptr() if self.gu[2] is not None else None,
            self.dn[0].data_ptr(), self.dn[1].data_ptr(), self.dn[2].data_ptr() if self.dn[2] is not None else None,
            ts, 1 if self.shared else 0,
            self.shared[0].desc if self.shared else empty, self.shared[1].desc if self.shared else empty)

    @property
    def nbytes_per_expert(self) -> int:
        tot = sum(t.numel() for t in self.gu if t is not None) + sum(t.numel() for t in self.dn if t is not None)
        return tot // self.n_experts


def route(logits, topk: int, workspace: Optional[Workspace] = None):
    """(topk_ids int32 [t, topk], topk_w fp32 [t, topk], route workspace) for fp32 logits [t, E] on the device."""
    import torch
    t, e = logits.shape
    ids = torch.empty((t, topk), dtype=torch.int32, device=logits.device)
    w = torch.empty((t, topk), dtype=torch.float32, device=logits.device)
    if workspace is None:
        workspace = Workspace(qmoe_route_workspace_size(t, e, topk), logits.device)
    qmoe_route(logits.data_ptr(), t, e, topk, ids.data_ptr(), w.data_ptr(), workspace.ptr, workspace.nbytes,
               _stream_ptr())
    return ids, w, workspace


def moe_ffn(pm: PackedMoE, x, topk_w, route_ws: Workspace, out=None, workspace: Optional[Workspace] = None,
            shared_gate=None):
    """One MoE FFN layer for the routed tokens x bf16 [t, H]: 1..4 tokens take the grouped-GEMV
    decode chain, more tokens the grouped tensor-core prefill chain.  shared_gate: fp32 [t]
    gate logits of the shared expert (its output is weighed by their sigmoid), or None."""
    import torch
    t = x.shape[0]
    topk = topk_w.shape[1]
    if out is None:
        out = torch.empty((t, (pm.hidden + 7) // 8 * 8), dtype=torch.bfloat16, device=x.device)[:, :pm.hidden]
    if workspace is None:
        workspace = Workspace(qmoe_workspace_size(pm.desc, t, topk), x.device)
    qmoe_ffn(pm.desc, x.data_ptr(), t, x.stride(0), topk, topk_w.data_ptr(),
             None if shared_gate is None else shared_gate.data_ptr(), route_ws.ptr, out.data_ptr(),
             out.stride(0), workspace.ptr, workspace.nbytes, _stream_ptr())
    return out


def moe_forward(pm: PackedMoE, x, logits, topk: int, out=None, workspace: Optional[Workspace] = None,
                route_ws: Optional[Workspace] = None, shared_gate=None):
    """Router and MoE FFN in one call (qmoe_forward) for x bf16 [t, H] and fp32 logits [t, E]:
    returns (out bf16 [t, H], topk_ids int32 [t, topk], topk_w fp32 [t, topk], route workspace)."""
    import torch
    t = x.shape[0]
    e = logits.shape[1]
    ids = torch.empty((t, topk), dtype=torch.int32, device=x.device)
    w = torch.empty((t, topk), dtype=torch.float32, device=x.device)
    if route_ws is None:
        route_ws = Workspace(qmoe_route_workspace_size(t, e, topk), x.device)
    if out is None:
        out = torch.empty((t, (pm.hidden + 7) // 8 * 8), dtype=torch.bfloat16, device=x.device)[:, :pm.hidden]
    if workspace is None:
        workspace = Workspace(qmoe_workspace_size(pm.desc, t, topk), x.device)
    qmoe_forward(pm.desc, x.data_ptr(), t, x.stride(0), logits.data_ptr(), topk,
                 None if shared_gate is None else shared_gate.data_ptr(), ids.data_ptr(), w.data_ptr(), route_ws.ptr,
                 route_ws.nbytes, out.data_ptr(), out.stride(0), workspace.ptr, workspace.nbytes, _stream_ptr())
    return out, ids, w, route_ws


def moe_stage(pm: PackedMoE, stage: int, inp, t: int, topk: int, route_ws: Workspace, topk_w=None, out=None,
              workspace: Optional[Workspace] = None, shared_gate=None):
    """One stage of the MoE FFN (qgemm_grouped): QG_MOE_GATE_UP_SWIGLU takes x bf16 [t, H] and
    returns h bf16 [t*topk + (t if shared), F] in the router's grouped row order;
    QG_MOE_DOWN_COMBINE takes that h, topk_w and optionally the shared expert's gate logits and
    returns out bf16 [t, H]."""
    import torch
    rows = t * topk + (t if pm.desc.has_shared else 0)
    cols = pm.ffn if stage == QG_MOE_GATE_UP_SWIGLU else pm.hidden
    n_out = rows if stage == QG_MOE_GATE_UP_SWIGLU else t
    if out is None:
        out = torch.empty((n_out, (cols + 7) // 8 * 8), dtype=torch.bfloat16, device=inp.device)[:, :cols]
    if workspace is None:
        workspace = Workspace(qgemm_grouped_workspace_size(pm.desc, t, topk, stage), inp.device)
    qgemm_grouped(pm.desc, stage, inp.data_ptr(), t, inp.stride(0), topk,
                  None if topk_w is None else topk_w.data_ptr(),
                  None if shared_gate is None else shared_gate.data_ptr(), route_ws.ptr, out.data_ptr(),
                  out.stride(0), workspace.ptr, workspace.nbytes, _stream_ptr())
    return out
