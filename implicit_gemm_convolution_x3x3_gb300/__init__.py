"""Python binding of the ig3 C ABI (include/ig3.h): fused stride-1 3x3(x3)
convolutions on GB300.

Argument marshalling only.  Every compute step runs in the CUDA kernels of
``_build/libig3.so``; PyTorch provides device memory and streams.  Importing
this package fails loudly when the library has not been built (there is no CPU
fallback): build it with ``python implicit_gemm_convolution_x3x3_gb300/build.py``.

The functions keep the C names: ``conv3d_fused``, ``dwsep_conv2d``,
``conv3d_fused_workspace_size``, ``conv3d_fused_select_path``,
``dwsep_conv2d_select_path``, ``ig3_status_string``, ``ig3_last_error``,
``ig3_last_device_status``, ``ig3_set_wait_timeout_ns``,
``ig3_selftest_bounded_wait``, ``ig3_kernel_launches``, ``ig3_version``.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libig3.so")

__all__ = [
    "EPILOGUES", "PATHS", "Ig3Error", "lib", "conv3d_fused", "dwsep_conv2d",
    "conv3d_fused_workspace_size", "conv3d_fused_select_path", "dwsep_conv2d_select_path",
    "dwsep_conv2d_ex_select_path",
    "conv3d_fused_noalloc", "NOALLOC_SCRATCH_BYTES",
    "ig3_status_string", "ig3_last_error", "ig3_last_device_status", "ig3_set_wait_timeout_ns",
    "ig3_selftest_bounded_wait", "ig3_kernel_launches", "ig3_version", "EXPORTED_SYMBOLS",
]

EPILOGUES = {"none": 0, "tanh_mish": 1, "pool_reduce": 2}
PATHS = {"auto": 0, "tc": 1, "fma": 2}
PATH_NAMES = {1: "tc", 2: "fma"}
NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024  # IG3_NOALLOC_SCRATCH_BYTES in include/ig3.h
STATUS = {0: "IG3_OK", -1: "IG3_ERR_INVALID_ARG", -2: "IG3_ERR_UNSUPPORTED", -3: "IG3_ERR_CUDA",
          -4: "IG3_ERR_TIMEOUT", -5: "IG3_ERR_WORKSPACE"}

if not os.path.exists(LIB_PATH):
    raise ImportError(f"the ig3 CUDA library is not built ({LIB_PATH} is missing); run "
                      "`python implicit_gemm_convolution_x3x3_gb300/build.py` first")

lib = ctypes.CDLL(LIB_PATH)

_i = ctypes.c_int
_p = ctypes.c_void_p
_sz = ctypes.c_size_t


class _EpiParams(ctypes.Structure):
    _fields_ = [("divisor", ctypes.c_float), ("pool", ctypes.c_int), ("bias2", ctypes.c_void_p)]


_SIGS = {
    "conv3d_fused_workspace_size": (_sz, [_i] * 8),
    "conv3d_fused": (_i, [_p, _i, _i, _i, _i, _i, _p, _i, _p, _i, ctypes.POINTER(_EpiParams), _p, _p, _sz,
                          _i, _p]),
    "conv3d_fused_noalloc": (_i, [_p, _i, _i, _i, _i, _i, _p, _i, _p, _i, ctypes.POINTER(_EpiParams), _p, _i,
                                  _p]),
    "dwsep_conv2d": (_i, [_p, _i, _i, _i, _i, _p, _p, _i, _p, _p, _i, _p]),
    "conv3d_fused_pad_workspace_size": (ctypes.c_size_t, [_i] * 9),
    "conv3d_fused_pad": (_i, [_p, _i, _i, _i, _i, _i, _i, _p, _i, _p, _i, _p, _p, _p, ctypes.c_size_t, _i, _p]),
    "conv3d_fused_ex_workspace_size": (ctypes.c_size_t, [_i] * 10),
    "conv3d_fused_ex": (_i, [_p, _i, _i, _i, _i, _i, _i, _i, _p, _i, _p, _i, _p, _p, _p, ctypes.c_size_t, _i, _p]),
    "dwsep_conv2d_ex": (_i, [_p, _i, _i, _i, _i, _i, _p, _p, _i, _p, _p, _i, _p]),
    "conv3d_fused_select_path": (_i, [_i] * 8),
    "dwsep_conv2d_select_path": (_i, [_i] * 6),
    "dwsep_conv2d_ex_select_path": (_i, [_i] * 7),
    "ig3_status_string": (ctypes.c_char_p, [_i]),
    "ig3_last_error": (ctypes.c_char_p, []),
    "ig3_last_device_status": (_i, [_p]),
    "ig3_set_wait_timeout_ns": (None, [ctypes.c_ulonglong]),
    "ig3_selftest_bounded_wait": (_i, [ctypes.c_ulonglong, _p]),
    "ig3_kernel_launches": (ctypes.c_ulonglong, []),
    "ig3_version": (ctypes.c_char_p, []),
}
EXPORTED_SYMBOLS = tuple(_SIGS)
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class Ig3Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def ig3_status_string(status: int) -> str:
    return lib.ig3_status_string(int(status)).decode()


def ig3_last_error() -> str:
    return lib.ig3_last_error().decode()


def ig3_version() -> str:
    return lib.ig3_version().decode()


def ig3_kernel_launches() -> int:
    return int(lib.ig3_kernel_launches())


def _check(status: int) -> None:
    if status != 0:
        raise Ig3Error(status, ig3_last_error())


def _stream_handle(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _dev_f32(t: torch.Tensor, name: str, shape=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def _enum(table, v, what):
    if isinstance(v, str):
        if v not in table:
            raise ValueError(f"unknown {what} {v!r}; one of {sorted(table)}")
        return table[v]
    return int(v)


def conv3d_fused_workspace_size(N, Cin, D, H, W, Cout, epilogue="tanh_mish", path="auto") -> int:
    return int(lib.conv3d_fused_workspace_size(N, Cin, D, H, W, Cout, _enum(EPILOGUES, epilogue, "epilogue"),
                                               _enum(PATHS, path, "path")))


def conv3d_fused_select_path(N, Cin, D, H, W, Cout, epilogue="tanh_mish", path="auto") -> str:
    r = lib.conv3d_fused_select_path(N, Cin, D, H, W, Cout, _enum(EPILOGUES, epilogue, "epilogue"),
                                     _enum(PATHS, path, "path"))
    _check(min(r, 0))
    return PATH_NAMES[r]


def dwsep_conv2d_select_path(N, C, H, W, Cout, path="auto") -> str:
    r = lib.dwsep_conv2d_select_path(N, C, H, W, Cout, _enum(PATHS, path, "path"))
    _check(min(r, 0))
    return PATH_NAMES[r]


def dwsep_conv2d_ex_select_path(N, C, H, W, K, Cout, path="auto") -> str:
    r = lib.dwsep_conv2d_ex_select_path(N, C, H, W, K, Cout, _enum(PATHS, path, "path"))
    _check(min(r, 0))
    return PATH_NAMES[r]


_workspaces: dict = {}


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    key = (device.type, device.index)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def conv3d_fused_pad_workspace_size(N, Cin, D, H, W, pad, Cout, epilogue="tanh_mish", path="auto") -> int:
    return int(lib.conv3d_fused_pad_workspace_size(N, Cin, D, H, W, pad, Cout,
                                                   _enum(EPILOGUES, epilogue, "epilogue"), _enum(PATHS, path, "path")))


def conv3d_fused_ex_workspace_size(N, Cin, D, H, W, pad, stride, Cout, epilogue="tanh_mish", path="auto") -> int:
    return int(lib.conv3d_fused_ex_workspace_size(N, Cin, D, H, W, pad, stride, Cout,
                                                  _enum(EPILOGUES, epilogue, "epilogue"), _enum(PATHS, path, "path")))


def conv3d_fused(x: torch.Tensor, w: torch.Tensor, b: torch.Tensor | None = None, epilogue="tanh_mish",
                 params: dict | None = None, out: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, path="auto", stream=None, pad: int = 0,
                 stride: int = 1) -> torch.Tensor:
    """3x3x3 conv3d with a fused epilogue (see include/ig3.h): valid, zero-padded by
    ``pad`` on every side (conv3d_fused_pad), or with stride 2 (conv3d_fused_ex).

    ``params`` (POOL_REDUCE only): ``{"divisor": 2.0, "pool": 2, "bias2": tensor[Cout]}``.
    Returns ``out`` ([N,Cout,OD,OH,OW] with OD = (D+2*pad-3)//stride+1, or [N] for POOL_REDUCE).
    """
    pad, stride = int(pad), int(stride)
    epi = _enum(EPILOGUES, epilogue, "epilogue")
    pth = _enum(PATHS, path, "path")
    if x.dim() != 5 or w.dim() != 5:
        raise ValueError("x must be [N,Cin,D,H,W] and w [Cout,Cin,3,3,3]")
    N, Cin, D, H, W = x.shape
    Cout = w.shape[0]
    xp = _dev_f32(x, "x")
    wp = _dev_f32(w, "w", (Cout, Cin, 3, 3, 3))
    bp = None if b is None else _dev_f32(b, "b", (Cout,))
    pr = None
    if epi == EPILOGUES["pool_reduce"]:
        params = params or {}
        if params.get("bias2") is None:
            raise ValueError("pool_reduce needs params['bias2']")
        pr = _EpiParams(float(params.get("divisor", 2.0)), int(params.get("pool", 2)),
                        _dev_f32(params["bias2"], "bias2", (Cout,)))
        oshape = (N,)
    else:
        oshape = (N, Cout) + tuple((s + 2 * pad - 3) // stride + 1 for s in (D, H, W))
    if out is None:
        out = torch.empty(oshape, dtype=torch.float32, device=x.device)
    yp = _dev_f32(out, "out", oshape)
    with torch.cuda.device(x.device):
        if stride != 1:
            need = int(lib.conv3d_fused_ex_workspace_size(N, Cin, D, H, W, pad, stride, Cout, epi, pth))
        elif pad == 0:
            need = int(lib.conv3d_fused_workspace_size(N, Cin, D, H, W, Cout, epi, pth))
        else:
            need = int(lib.conv3d_fused_pad_workspace_size(N, Cin, D, H, W, pad, Cout, epi, pth))
        if workspace is None and need > 0:
            workspace = _workspace(x.device, need)
        wsp = None if workspace is None else workspace.data_ptr()
        wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
        epp = None if pr is None else ctypes.byref(pr)
        if stride != 1:
            st = lib.conv3d_fused_ex(xp, N, Cin, D, H, W, pad, stride, wp, Cout, bp, epi, epp, yp, wsp, wsb, pth,
                                     _stream_handle(stream, x.device))
        elif pad == 0:
            st = lib.conv3d_fused(xp, N, Cin, D, H, W, wp, Cout, bp, epi, epp, yp, wsp, wsb, pth,
                                  _stream_handle(stream, x.device))
        else:
            st = lib.conv3d_fused_pad(xp, N, Cin, D, H, W, pad, wp, Cout, bp, epi, epp, yp, wsp, wsb, pth,
                                      _stream_handle(stream, x.device))
    _check(st)
    return out


def conv3d_fused_noalloc(x: torch.Tensor, w: torch.Tensor, b: torch.Tensor | None = None,
                         epilogue="tanh_mish", params: dict | None = None, out: torch.Tensor | None = None,
                         path="auto", stream=None) -> torch.Tensor:
    """conv3d_fused with the scratch taken from the library's static buffer.

    For callers that cannot allocate device memory per call.  ``out`` must be given
    for the call itself to allocate nothing (else it is created here with torch).
    See include/ig3.h for the buffer size, the first-call set-up and the rule that
    calls overlapping on the GPU race on the shared buffer.
    """
    epi = _enum(EPILOGUES, epilogue, "epilogue")
    pth = _enum(PATHS, path, "path")
    if x.dim() != 5 or w.dim() != 5:
        raise ValueError("x must be [N,Cin,D,H,W] and w [Cout,Cin,3,3,3]")
    N, Cin, D, H, W = x.shape
    Cout = w.shape[0]
    xp = _dev_f32(x, "x")
    wp = _dev_f32(w, "w", (Cout, Cin, 3, 3, 3))
    bp = None if b is None else _dev_f32(b, "b", (Cout,))
    pr = None
    if epi == EPILOGUES["pool_reduce"]:
        params = params or {}
        if params.get("bias2") is None:
            raise ValueError("pool_reduce needs params['bias2']")
        pr = _EpiParams(float(params.get("divisor", 2.0)), int(params.get("pool", 2)),
                        _dev_f32(params["bias2"], "bias2", (Cout,)))
        oshape = (N,)
    else:
        oshape = (N, Cout, D - 2, H - 2, W - 2)
    if out is None:
        out = torch.empty(oshape, dtype=torch.float32, device=x.device)
    yp = _dev_f32(out, "out", oshape)
    with torch.cuda.device(x.device):
        st = lib.conv3d_fused_noalloc(xp, N, Cin, D, H, W, wp, Cout, bp, epi,
                                      None if pr is None else ctypes.byref(pr), yp, pth,
                                      _stream_handle(stream, x.device))
    _check(st)
    return out


def dwsep_conv2d(x: torch.Tensor, w_dw: torch.Tensor, w_pw: torch.Tensor, b: torch.Tensor | None = None,
                 out: torch.Tensor | None = None, path="auto", stream=None) -> torch.Tensor:
    """Depthwise KxK ("same" padding (K-1)/2; K = w_dw.shape[-1], 3 by the source problem)
    then pointwise 1x1 conv2d (see include/ig3.h); returns [N,Cout,H,W]."""
    pth = _enum(PATHS, path, "path")
    if x.dim() != 4 or w_dw.dim() != 4:
        raise ValueError("x must be [N,C,H,W] and w_dw [C,1,K,K]")
    N, C, H, W = x.shape
    K = int(w_dw.shape[-1])
    Cout = w_pw.shape[0]
    xp = _dev_f32(x, "x")
    dp = _dev_f32(w_dw, "w_dw", (C, 1, K, K))
    pp = _dev_f32(w_pw, "w_pw", (Cout, C, 1, 1))
    bp = None if b is None else _dev_f32(b, "b", (Cout,))
    if out is None:
        out = torch.empty((N, Cout, H, W), dtype=torch.float32, device=x.device)
    yp = _dev_f32(out, "out", (N, Cout, H, W))
    with torch.cuda.device(x.device):
        if K == 3:
            st = lib.dwsep_conv2d(xp, N, C, H, W, dp, pp, Cout, bp, yp, pth, _stream_handle(stream, x.device))
        else:
            st = lib.dwsep_conv2d_ex(xp, N, C, H, W, K, dp, pp, Cout, bp, yp, pth, _stream_handle(stream, x.device))
    _check(st)
    return out


def ig3_last_device_status(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device status: 0 or IG3_ERR_TIMEOUT."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib.ig3_last_device_status(_stream_handle(stream, dev)))


def ig3_set_wait_timeout_ns(ns: int) -> None:
    lib.ig3_set_wait_timeout_ns(int(ns))


def ig3_selftest_bounded_wait(timeout_ns: int, stream=None, device=None) -> None:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib.ig3_selftest_bounded_wait(int(timeout_ns), _stream_handle(stream, dev)))
