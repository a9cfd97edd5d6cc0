"""CPU float64 oracle for the fused 3x3(x3) convolutions.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
(the CUDA library and its Python binding) never imports or calls it, and this
package imports nothing from the product.

The arithmetic lives in ``ig3_oracle.c`` (plain nested loops, float64
accumulation); this module compiles it with gcc on first use and wraps it with
numpy-facing functions.  Every function returns float64.

Parity status of each function (what pins it; see tests/test_oracle_pins.py):
  conv3d / conv3d_at       pinned: brute-force im2col x W^T, scipy correlate,
                           delta kernel, constant input, linearity, translation.
  conv3d_pad / _at         pinned: np.pad + brute-force im2col, scipy correlate in
                           'same' mode, delta kernel (y = x), constant-input corner and
                           interior closed forms, pad 0 == conv3d.
  conv3d_ex / _at          pinned: np.pad + strided brute-force im2col, scipy valid
                           correlation subsampled, centre delta with stride 2 (y =
                           x[::2]), stride 1 == conv3d_pad, the printed size formula.
  tanh_mish                pinned: algebraic identity form, special values,
                           large-y asymptote, Mish minimum.
  pool_reduce              pinned: window enumeration, S/(div*cells)+sum(bias2)
                           identity, constant input, floor mode, planted maxima.
  dwsep / dwsep_single_sum pinned: scipy correlate2d + einsum, two-stage ==
                           single-sum, centre-delta and identity special cases.
  dwsep_k / dwsep_k_at     pinned: scipy correlate2d 'same' + einsum for K = 1, 3, 5,
                           7, two-stage == single-sum, K = 3 == dwsep, centre delta.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ig3_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libig3_oracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_fp = ctypes.POINTER(ctypes.c_float)
_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (OpenMP, strict IEEE float)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_conv3d_at.restype = ctypes.c_double
        lib.oracle_conv3d_at.argtypes = [_fp, _i64, _i64, _i64, _i64, _i64, _fp, _i64, _fp,
                                         _i64, _i64, _i64, _i64, _i64]
        lib.oracle_conv3d.restype = None
        lib.oracle_conv3d.argtypes = [_fp, _i64, _i64, _i64, _i64, _i64, _fp, _i64, _fp, _dp]
        lib.oracle_conv3d_pad_at.restype = ctypes.c_double
        lib.oracle_conv3d_pad_at.argtypes = [_fp, _i64, _i64, _i64, _i64, _i64, _i64, _fp, _i64, _fp,
                                             _i64, _i64, _i64, _i64, _i64]
        lib.oracle_conv3d_ex_at.restype = ctypes.c_double
        lib.oracle_conv3d_ex_at.argtypes = [_fp, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _fp, _i64, _fp,
                                            _i64, _i64, _i64, _i64, _i64]
        lib.oracle_conv3d_ex.restype = None
        lib.oracle_conv3d_ex.argtypes = [_fp, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _fp, _i64, _fp, _dp]
        lib.oracle_dwsep_k.restype = ctypes.c_int
        lib.oracle_dwsep_k.argtypes = [_fp, _i64, _i64, _i64, _i64, _i64, _fp, _fp, _i64, _fp, _dp]
        lib.oracle_dwsep_k_at.restype = ctypes.c_double
        lib.oracle_dwsep_k_at.argtypes = [_fp, _i64, _i64, _i64, _i64, _i64, _fp, _fp, _i64, _fp,
                                          _i64, _i64, _i64, _i64]
        lib.oracle_conv3d_pad.restype = None
        lib.oracle_conv3d_pad.argtypes = [_fp, _i64, _i64, _i64, _i64, _i64, _i64, _fp, _i64, _fp, _dp]
        lib.oracle_tanh_mish.restype = ctypes.c_double
        lib.oracle_tanh_mish.argtypes = [ctypes.c_double]
        lib.oracle_tanh_mish_array.restype = None
        lib.oracle_tanh_mish_array.argtypes = [_dp, _i64, _dp]
        lib.oracle_pool_reduce.restype = None
        lib.oracle_pool_reduce.argtypes = [_dp, _i64, _i64, _i64, _i64, _i64, ctypes.c_double,
                                           _i64, _fp, _dp]
        lib.oracle_dwsep.restype = ctypes.c_int
        lib.oracle_dwsep.argtypes = [_fp, _i64, _i64, _i64, _i64, _fp, _fp, _i64, _fp, _dp]
        lib.oracle_dwsep_at.restype = ctypes.c_double
        lib.oracle_dwsep_at.argtypes = [_fp, _i64, _i64, _i64, _i64, _fp, _fp, _i64, _fp,
                                        _i64, _i64, _i64, _i64]
        lib.oracle_dwsep_single_sum.restype = None
        lib.oracle_dwsep_single_sum.argtypes = [_fp, _i64, _i64, _i64, _i64, _fp, _fp, _i64,
                                                _fp, _dp]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    if not np.all(np.isfinite(a)):
        raise ValueError("oracle inputs must be finite")
    return a


def _fptr(a):
    return None if a is None else a.ctypes.data_as(_fp)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


# ---------------------------------------------------------------- shapes / counts
def conv3d_out_dims(D: int, H: int, W: int) -> tuple:
    """Valid stride-1 k=3 output size: each spatial dim shrinks by 3 - 1 = 2."""
    return (D - 3 + 1, H - 3 + 1, W - 3 + 1)


def pooled_dims(OD: int, OH: int, OW: int, pool: int = 2) -> tuple:
    """MaxPool3d(pool, stride=pool, floor mode) output size."""
    return ((OD - pool) // pool + 1, (OH - pool) // pool + 1, (OW - pool) // pool + 1)


def conv3d_macs(N, Cin, D, H, W, Cout) -> int:
    OD, OH, OW = conv3d_out_dims(D, H, W)
    return N * Cout * OD * OH * OW * Cin * 27


def dwsep_macs(N, C, H, W, Cout) -> int:
    return N * H * W * C * (9 + Cout)


# ---------------------------------------------------------------- conv3d
def conv3d(x, w, b=None) -> np.ndarray:
    """Valid stride-1 3x3x3 cross-correlation, float64 result [N,Cout,D-2,H-2,W-2]."""
    lib = _load()
    x = _f32(x); w = _f32(w); b = None if b is None else _f32(b)
    N, Cin, D, H, W = x.shape
    Cout = w.shape[0]
    assert w.shape == (Cout, Cin, 3, 3, 3)
    OD, OH, OW = conv3d_out_dims(D, H, W)
    y = np.empty((N, Cout, max(OD, 0), max(OH, 0), max(OW, 0)), dtype=np.float64)
    lib.oracle_conv3d(_fptr(x), N, Cin, D, H, W, _fptr(w), Cout, _fptr(b),
                      y.ctypes.data_as(_dp))
    return y


def conv3d_at(x, w, b, index) -> np.ndarray:
    """Conv outputs at a list of (n, k, od, oh, ow) indices (float64)."""
    lib = _load()
    x = _f32(x); w = _f32(w); b = None if b is None else _f32(b)
    N, Cin, D, H, W = x.shape
    Cout = w.shape[0]
    idx = np.asarray(index, dtype=np.int64).reshape(-1, 5)
    out = np.empty(len(idx), dtype=np.float64)
    xp, wp, bp = _fptr(x), _fptr(w), _fptr(b)
    for i, (n, k, od, oh, ow) in enumerate(idx):
        out[i] = lib.oracle_conv3d_at(xp, N, Cin, D, H, W, wp, Cout, bp,
                                      int(n), int(k), int(od), int(oh), int(ow))
    return out


def conv3d_pad(x, w, b=None, pad: int = 1) -> np.ndarray:
    """Zero-padded stride-1 3x3x3 cross-correlation, float64 [N,Cout,D+2P-2,H+2P-2,W+2P-2]."""
    lib = _load()
    x = _f32(x); w = _f32(w); b = None if b is None else _f32(b)
    N, Cin, D, H, W = x.shape
    Cout = w.shape[0]
    assert w.shape == (Cout, Cin, 3, 3, 3) and pad >= 0
    OD, OH, OW = D + 2 * pad - 2, H + 2 * pad - 2, W + 2 * pad - 2
    y = np.empty((N, Cout, max(OD, 0), max(OH, 0), max(OW, 0)), dtype=np.float64)
    lib.oracle_conv3d_pad(_fptr(x), N, Cin, D, H, W, int(pad), _fptr(w), Cout, _fptr(b),
                          y.ctypes.data_as(_dp))
    return y


def conv3d_pad_at(x, w, b, pad: int, index) -> np.ndarray:
    """Padded conv outputs at a list of (n, k, od, oh, ow) indices (float64)."""
    lib = _load()
    x = _f32(x); w = _f32(w); b = None if b is None else _f32(b)
    N, Cin, D, H, W = x.shape
    Cout = w.shape[0]
    idx = np.asarray(index, dtype=np.int64).reshape(-1, 5)
    out = np.empty(len(idx), dtype=np.float64)
    xp, wp, bp = _fptr(x), _fptr(w), _fptr(b)
    for i, (n, k, od, oh, ow) in enumerate(idx):
        out[i] = lib.oracle_conv3d_pad_at(xp, N, Cin, D, H, W, int(pad), wp, Cout, bp,
                                          int(n), int(k), int(od), int(oh), int(ow))
    return out


def conv3d_ex_out_dims(D: int, H: int, W: int, pad: int, stride: int) -> tuple:
    return tuple((s + 2 * pad - 3) // stride + 1 for s in (D, H, W))


def conv3d_ex(x, w, b=None, pad: int = 0, stride: int = 1) -> np.ndarray:
    """Zero-padded 3x3x3 cross-correlation with stride, float64 [N,Cout,OD,OH,OW]."""
    lib = _load()
    x = _f32(x); w = _f32(w); b = None if b is None else _f32(b)
    N, Cin, D, H, W = x.shape
    Cout = w.shape[0]
    assert w.shape == (Cout, Cin, 3, 3, 3) and pad >= 0 and stride >= 1
    OD, OH, OW = conv3d_ex_out_dims(D, H, W, pad, stride)
    y = np.empty((N, Cout, max(OD, 0), max(OH, 0), max(OW, 0)), dtype=np.float64)
    lib.oracle_conv3d_ex(_fptr(x), N, Cin, D, H, W, int(pad), int(stride), _fptr(w), Cout, _fptr(b),
                         y.ctypes.data_as(_dp))
    return y


def conv3d_ex_at(x, w, b, pad: int, stride: int, index) -> np.ndarray:
    """Strided, padded conv outputs at a list of (n, k, od, oh, ow) indices (float64)."""
    lib = _load()
    x = _f32(x); w = _f32(w); b = None if b is None else _f32(b)
    N, Cin, D, H, W = x.shape
    Cout = w.shape[0]
    idx = np.asarray(index, dtype=np.int64).reshape(-1, 5)
    out = np.empty(len(idx), dtype=np.float64)
    xp, wp, bp = _fptr(x), _fptr(w), _fptr(b)
    for i, (n, k, od, oh, ow) in enumerate(idx):
        out[i] = lib.oracle_conv3d_ex_at(xp, N, Cin, D, H, W, int(pad), int(stride), wp, Cout, bp,
                                         int(n), int(k), int(od), int(oh), int(ow))
    return out


def tanh_mish(y) -> np.ndarray:
    """tanh(y * tanh(log1p(exp(y)))) elementwise in float64."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.float64)
    out = np.empty_like(y)
    lib.oracle_tanh_mish_array(y.ctypes.data_as(_dp), y.size, out.ctypes.data_as(_dp))
    return out


def tanh_mish_scalar(y: float) -> float:
    return _load().oracle_tanh_mish(float(y))


def pool_reduce(y, divisor: float, pool: int, bias2) -> np.ndarray:
    """/divisor -> maxpool(pool, floor) -> global mean -> +bias2[c] -> sum over c; out[N]."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.float64)
    bias2 = _f32(bias2)
    N, C, OD, OH, OW = y.shape
    assert bias2.shape == (C,)
    out = np.empty(N, dtype=np.float64)
    lib.oracle_pool_reduce(y.ctypes.data_as(_dp), N, C, OD, OH, OW, float(divisor), int(pool),
                           _fptr(bias2), out.ctypes.data_as(_dp))
    return out


def conv3d_tanh_mish(x, w, b) -> np.ndarray:
    return tanh_mish(conv3d(x, w, b))


def conv3d_pool_reduce(x, w, b, divisor: float, pool: int, bias2) -> np.ndarray:
    return pool_reduce(conv3d(x, w, b), divisor, pool, bias2)


# ---------------------------------------------------------------- dwsep
def dwsep(x, w_dw, w_pw, b=None) -> np.ndarray:
    """Depthwise 3x3 (pad 1) then pointwise 1x1, two-stage, float64 [N,Cout,H,W]."""
    lib = _load()
    x = _f32(x); w_dw = _f32(w_dw); w_pw = _f32(w_pw); b = None if b is None else _f32(b)
    N, C, H, W = x.shape
    Cout = w_pw.shape[0]
    assert w_dw.shape == (C, 1, 3, 3) and w_pw.shape == (Cout, C, 1, 1)
    out = np.empty((N, Cout, H, W), dtype=np.float64)
    rc = lib.oracle_dwsep(_fptr(x), N, C, H, W, _fptr(w_dw), _fptr(w_pw), Cout, _fptr(b),
                          out.ctypes.data_as(_dp))
    if rc != 0:
        raise MemoryError("oracle_dwsep could not allocate its depthwise stage")
    return out


def dwsep_single_sum(x, w_dw, w_pw, b=None) -> np.ndarray:
    lib = _load()
    x = _f32(x); w_dw = _f32(w_dw); w_pw = _f32(w_pw); b = None if b is None else _f32(b)
    N, C, H, W = x.shape
    Cout = w_pw.shape[0]
    out = np.empty((N, Cout, H, W), dtype=np.float64)
    lib.oracle_dwsep_single_sum(_fptr(x), N, C, H, W, _fptr(w_dw), _fptr(w_pw), Cout, _fptr(b),
                                out.ctypes.data_as(_dp))
    return out


def dwsep_k(x, w_dw, w_pw, b=None) -> np.ndarray:
    """Depthwise KxK ("same" padding (K-1)/2, K odd) then pointwise 1x1, two-stage, float64."""
    lib = _load()
    x = _f32(x); w_dw = _f32(w_dw); w_pw = _f32(w_pw); b = None if b is None else _f32(b)
    N, C, H, W = x.shape
    K = w_dw.shape[-1]
    Cout = w_pw.shape[0]
    assert w_dw.shape == (C, 1, K, K) and K % 2 == 1 and w_pw.shape == (Cout, C, 1, 1)
    out = np.empty((N, Cout, H, W), dtype=np.float64)
    if lib.oracle_dwsep_k(_fptr(x), N, C, H, W, K, _fptr(w_dw), _fptr(w_pw), Cout, _fptr(b),
                          out.ctypes.data_as(_dp)) != 0:
        raise MemoryError("oracle_dwsep_k could not allocate its depthwise stage")
    return out


def dwsep_k_at(x, w_dw, w_pw, b, index) -> np.ndarray:
    """dwsep_k outputs at a list of (n, o, h, w) indices (single-sum form, float64)."""
    lib = _load()
    x = _f32(x); w_dw = _f32(w_dw); w_pw = _f32(w_pw); b = None if b is None else _f32(b)
    N, C, H, W = x.shape
    K = w_dw.shape[-1]
    Cout = w_pw.shape[0]
    idx = np.asarray(index, dtype=np.int64).reshape(-1, 4)
    out = np.empty(len(idx), dtype=np.float64)
    xp, dp_, pp, bp = _fptr(x), _fptr(w_dw), _fptr(w_pw), _fptr(b)
    for i, (n, o, h, w) in enumerate(idx):
        out[i] = lib.oracle_dwsep_k_at(xp, N, C, H, W, K, dp_, pp, Cout, bp, int(n), int(o), int(h), int(w))
    return out


def dwsep_at(x, w_dw, w_pw, b, index) -> np.ndarray:
    """dwsep outputs at a list of (n, o, h, w) indices (float64)."""
    lib = _load()
    x = _f32(x); w_dw = _f32(w_dw); w_pw = _f32(w_pw); b = None if b is None else _f32(b)
    N, C, H, W = x.shape
    Cout = w_pw.shape[0]
    idx = np.asarray(index, dtype=np.int64).reshape(-1, 4)
    out = np.empty(len(idx), dtype=np.float64)
    xp, dp_, pp, bp = _fptr(x), _fptr(w_dw), _fptr(w_pw), _fptr(b)
    for i, (n, o, h, w) in enumerate(idx):
        out[i] = lib.oracle_dwsep_at(xp, N, C, H, W, dp_, pp, Cout, bp,
                                     int(n), int(o), int(h), int(w))
    return out
