"""The C-ABI library without a GPU: it loads, exports every symbol include/ig3.h
declares, and rejects bad arguments with status codes before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ig3.h")


def _build_if_needed():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "ig3_build", os.path.join(ROOT, "implicit_gemm_convolution_x3x3_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


@pytest.fixture(scope="module")
def lib():
    path = _build_if_needed()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\(", text)) - {"defined"})


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ("conv3d_fused", "dwsep_conv2d", "ig3_status_string", "ig3_last_device_status",
              "conv3d_fused_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared in ig3.h but not exported"


def test_python_binding_lists_every_symbol():
    import sys
    sys.path.insert(0, ROOT)
    torch = pytest.importorskip("torch")  # noqa: F841  (the binding imports torch)
    _build_if_needed()
    import implicit_gemm_convolution_x3x3_gb300 as m
    assert sorted(m.EXPORTED_SYMBOLS) == declared_functions()


def test_noalloc_scratch_size_matches_header():
    # The binding's NOALLOC_SCRATCH_BYTES is what the tests size their shapes by: it
    # must be the header's IG3_NOALLOC_SCRATCH_BYTES, the size of the library's buffer.
    import sys
    sys.path.insert(0, ROOT)
    pytest.importorskip("torch")
    _build_if_needed()
    import implicit_gemm_convolution_x3x3_gb300 as m
    text = open(HEADER).read()
    mt = re.search(r"#define\s+IG3_NOALLOC_SCRATCH_BYTES\s+\(([^)]*)\)", text)
    assert mt, "IG3_NOALLOC_SCRATCH_BYTES not found in ig3.h"
    expr = mt.group(1).replace("u", "")
    assert re.fullmatch(r"[0-9*+ ]+", expr), expr
    assert eval(expr) == m.NOALLOC_SCRATCH_BYTES


def _c(lib):
    f = lib.conv3d_fused
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    return f


class EpiParams(ctypes.Structure):
    _fields_ = [("divisor", ctypes.c_float), ("pool", ctypes.c_int), ("bias2", ctypes.c_void_p)]


FAKE = 4096  # never dereferenced: every case below fails host-side validation first


def test_status_strings(lib):
    lib.ig3_status_string.restype = ctypes.c_char_p
    assert lib.ig3_status_string(0) == b"IG3_OK"
    assert lib.ig3_status_string(-4) == b"IG3_ERR_TIMEOUT"
    assert lib.ig3_status_string(-5) == b"IG3_ERR_WORKSPACE"
    assert lib.ig3_status_string(12) == b"IG3_ERR_UNKNOWN"


@pytest.mark.parametrize("args,status", [
    ((1, 1, 3, 3, 3, 1, 0, 0), 0),       # valid (checked below only for the error cases)
    ((0, 1, 3, 3, 3, 1, 1, 0), -1),      # N = 0
    ((1, -2, 3, 3, 3, 1, 1, 0), -1),     # Cin < 0
    ((1, 1, 2, 3, 3, 1, 1, 0), -2),      # D < 3: no valid output
    ((1, 1, 3, 3, 3, 1, 7, 0), -1),      # unknown epilogue
    ((1, 1, 3, 3, 3, 1, 1, 9), -1),      # unknown path
    ((1, 1, 3, 3, 3, 2, 1, 1), -2),      # TC path with Cout = 2
    ((4096, 64, 64, 64, 64, 64, 1, 0), -1),  # 2^31 or more elements
    ((1, 1, 3, 3, 3, 1, 2, 0), -2),      # pool-reduce with an empty pooled grid
])
def test_conv3d_argument_errors(lib, args, status):
    f = lib.conv3d_fused_select_path
    f.restype = ctypes.c_int
    r = f(*args)
    if status == 0:
        assert r in (1, 2)
    else:
        assert r == status
        conv = _c(lib)
        N, Cin, D, H, W, Cout, epi, path = args
        assert conv(FAKE, N, Cin, D, H, W, FAKE, Cout, None, epi, None, FAKE, None, 0, path, None) == status
        lib.ig3_last_error.restype = ctypes.c_char_p
        assert len(lib.ig3_last_error()) > 0


@pytest.mark.parametrize("args,expected", [
    ((1, 1, 3, 3, 4, 16, 1), 1),          # the smallest measured shape: tensor cores (8.7 vs 13.0 us)
    ((2, 4, 8, 8, 8, 16, 1), 1),
    ((16, 32, 32, 64, 64, 64, 1), 1),     # the conv3d + tanh(mish) workload
    ((128, 8, 16, 64, 64, 16, 2), 1),     # the pool-reduce workload
    ((2, 4, 8, 8, 8, 8, 1), 2),           # Cout 8: no tensor-core kernel
    ((1, 8, 5, 7, 9, 144, 0), 2),         # Cout above 128
    ((1, 8, 6, 8, 13, 16, 2), 2),         # pool-reduce with W not dividing 64
])
def test_conv3d_automatic_path_choice(lib, args, expected):
    # The automatic choice follows the measured crossover: tensor cores wherever a
    # tensor-core kernel covers the shape, the FMA kernel elsewhere (1 = TC, 2 = FMA).
    f = lib.conv3d_fused_select_path
    f.restype = ctypes.c_int
    assert f(*args, 0) == expected


def test_conv3d_null_and_param_errors(lib):
    conv = _c(lib)
    assert conv(None, 1, 1, 3, 3, 3, FAKE, 1, None, 1, None, FAKE, None, 0, 2, None) == -1
    # pool-reduce needs params with bias2, pool == 2 and a finite nonzero divisor
    assert conv(FAKE, 1, 1, 4, 4, 4, FAKE, 1, None, 2, None, FAKE, None, 0, 2, None) == -1
    p = EpiParams(2.0, 3, FAKE)
    assert conv(FAKE, 1, 1, 4, 4, 4, FAKE, 1, None, 2, ctypes.byref(p), FAKE, None, 0, 2, None) == -2
    p = EpiParams(0.0, 2, FAKE)
    assert conv(FAKE, 1, 1, 4, 4, 4, FAKE, 1, None, 2, ctypes.byref(p), FAKE, None, 0, 2, None) == -1
    p = EpiParams(float("inf"), 2, FAKE)
    assert conv(FAKE, 1, 1, 4, 4, 4, FAKE, 1, None, 2, ctypes.byref(p), FAKE, None, 0, 2, None) == -1
    # a needed workspace that is missing, too small or misaligned
    lib.conv3d_fused_workspace_size.restype = ctypes.c_size_t
    need = lib.conv3d_fused_workspace_size(1, 1, 4, 4, 4, 1, 2, 2)
    assert need > 0
    p = EpiParams(2.0, 2, FAKE)
    assert conv(FAKE, 1, 1, 4, 4, 4, FAKE, 1, None, 2, ctypes.byref(p), FAKE, None, 0, 2, None) == -5
    assert conv(FAKE, 1, 1, 4, 4, 4, FAKE, 1, None, 2, ctypes.byref(p), FAKE, FAKE, need - 1, 2, None) == -5
    assert conv(FAKE, 1, 1, 4, 4, 4, FAKE, 1, None, 2, ctypes.byref(p), FAKE, FAKE + 4, need, 2, None) == -5


def test_dwsep_argument_errors(lib):
    f = lib.dwsep_conv2d
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2 + [ctypes.c_int] + \
        [ctypes.c_void_p] * 2 + [ctypes.c_int, ctypes.c_void_p]
    assert f(FAKE, 0, 4, 5, 5, FAKE, FAKE, 4, None, FAKE, 2, None) == -1
    assert f(FAKE, 1, 4, 5, 5, FAKE, FAKE, 4, None, FAKE, 5, None) == -1
    assert f(None, 1, 4, 5, 5, FAKE, FAKE, 4, None, FAKE, 2, None) == -1
    assert f(FAKE, 1, 4, 5, 5, FAKE, FAKE, 4, None, FAKE, 1, None) == -2   # TC: Cout = 4
    assert f(FAKE, 70000, 64, 512, 512, FAKE, FAKE, 4, None, FAKE, 2, None) == -1  # too many elements


def test_workspace_query_is_zero_for_rejected_args(lib):
    lib.conv3d_fused_workspace_size.restype = ctypes.c_size_t
    assert lib.conv3d_fused_workspace_size(0, 1, 3, 3, 3, 1, 1, 0) == 0
    assert lib.conv3d_fused_workspace_size(1, 1, 3, 3, 3, 1, 1, 2) == 0  # tanh-mish on FMA needs none


def _pad(lib):
    f = lib.conv3d_fused_pad
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 6 + [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                                           ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                                           ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                                           ctypes.c_void_p]
    return f


def test_conv3d_pad_argument_errors(lib):
    f = _pad(lib)
    q = lib.conv3d_fused_pad_workspace_size
    q.restype = ctypes.c_size_t
    # pad out of range, non-positive dims, too many padded elements: rejected before any launch
    assert f(FAKE, 1, 1, 3, 3, 3, -1, FAKE, 1, None, 1, None, FAKE, FAKE, 1 << 20, 2, None) == -1
    assert f(FAKE, 1, 1, 3, 3, 3, 17, FAKE, 1, None, 1, None, FAKE, FAKE, 1 << 20, 2, None) == -1
    assert f(FAKE, 1, 1, 0, 3, 3, 1, FAKE, 1, None, 1, None, FAKE, FAKE, 1 << 20, 2, None) == -1
    assert f(FAKE, 2048, 64, 62, 62, 62, 1, FAKE, 1, None, 1, None, FAKE, FAKE, 1 << 20, 2, None) == -1
    # the TC path's own requirements apply to the padded shape (Cout = 2)
    assert f(FAKE, 1, 1, 3, 3, 3, 1, FAKE, 2, None, 1, None, FAKE, FAKE, 1 << 20, 1, None) == -2
    # the border is never materialised: a padded call needs only the valid path's workspace
    need = q(1, 16, 4, 5, 6, 1, 16, 1, 1)        # tensor cores: the split weights
    assert need > 0 and need % 256 == 0
    assert need <= lib.conv3d_fused_workspace_size(1, 16, 6, 7, 8, 16, 1, 1) + 256 * 1024
    assert f(FAKE, 1, 16, 4, 5, 6, 1, FAKE, 16, None, 1, None, FAKE, None, 0, 1, None) == -5
    assert f(FAKE, 1, 16, 4, 5, 6, 1, FAKE, 16, None, 1, None, FAKE, FAKE, need - 1, 1, None) == -5
    assert f(FAKE, 1, 16, 4, 5, 6, 1, FAKE, 16, None, 1, None, FAKE, FAKE + 4, need, 1, None) == -5
    assert q(1, 1, 1, 1, 1, 1, 1, 1, 2) == 0   # FMA path, tanh(mish): no workspace at all
    # the padded conv3d + tanh(mish) workload: a few hundred KB of split weights, where the
    # zero-bordered copy of x alone would be 303 MB
    lib.conv3d_fused_workspace_size.restype = ctypes.c_size_t
    assert 0 < q(16, 32, 32, 64, 64, 1, 64, 1, 1) < (1 << 20)
    # queries: zero for rejected arguments; pad 0 is the valid-conv query
    assert q(1, 1, 3, 3, 3, -1, 1, 1, 2) == 0
    assert q(0, 1, 3, 3, 3, 1, 1, 1, 2) == 0
    assert q(1, 1, 4, 4, 4, 0, 1, 2, 2) == lib.conv3d_fused_workspace_size(1, 1, 4, 4, 4, 1, 2, 2)


def test_dwsep_auto_path_follows_measured_crossover(lib):
    # Shapes from the measured crossover of the two depthwise-separable paths
    # (bench.py --study dwsep_crossover): the faster path there is the automatic choice.
    f = lib.dwsep_conv2d_select_path
    f.restype = ctypes.c_int
    TC, FMA = 1, 2
    assert f(1, 16, 32, 32, 128, 0) == FMA     # tiny, C = 16: FMA 13.9 us, TC 23.5 us
    assert f(2, 64, 128, 128, 16, 0) == TC     # TC 23.5 us, FMA 33.3 us
    assert f(1, 64, 64, 64, 32, 0) == TC       # TC 25.2 us, FMA 33.3 us
    assert f(4, 64, 256, 256, 128, 0) == TC    # TC 60 us, FMA 458 us
    assert f(1, 24, 64, 64, 32, 0) == FMA      # C not a multiple of 16: no TC kernel


def test_conv3d_ex_argument_errors(lib):
    f = lib.conv3d_fused_ex
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                                           ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                                           ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                                           ctypes.c_void_p]
    q = lib.conv3d_fused_ex_workspace_size
    q.restype = ctypes.c_size_t
    args = lambda D, pad, stride, Cout, epi, path, x=FAKE: (x, 1, 2, D, D, D, pad, stride, FAKE, Cout, None, epi,
                                                          None, FAKE, None, 0, path, None)
    assert f(*args(5, 1, 3, 4, 1, 0)) == -2       # stride 3: not built
    assert f(*args(5, 1, 0, 4, 1, 0)) == -2       # stride 0
    assert f(*args(5, -1, 2, 4, 1, 0)) == -1      # negative pad
    assert f(*args(5, 1, 2, 4, 2, 0)) == -2       # stride 2 with pool-reduce
    assert f(*args(5, 1, 2, 16, 1, 1)) == -2      # stride 2 on the TC path, W not a multiple of 4
    assert f(*args(5, 1, 2, 8, 1, 1)) == -2       # stride 2 on the TC path, Cout not a multiple of 16
    assert f(*args(2, 0, 2, 4, 1, 0)) == -2       # no output (D + 2*pad < 3)
    assert f(*args(5, 1, 2, 4, 1, 0, None)) == -1  # NULL x
    assert q(1, 2, 5, 5, 5, 1, 2, 4, 1, 0) == 0   # stride 2 on the FMA kernel needs no workspace
    # stride 2 on tensor cores: the split weight blocks, 3 kd x K-steps x 576 * Cout bytes
    assert q(1, 32, 32, 64, 64, 1, 2, 64, 1, 0) == 3 * 4 * 576 * 64
    assert q(1, 32, 32, 64, 64, 1, 2, 64, 1, 2) == 0   # forced FMA
    assert q(1, 32, 32, 64, 64, 1, 2, 64, 2, 0) == 0   # pool-reduce: not with stride 2
    assert q(1, 2, 5, 5, 5, 1, 1, 16, 1, 1) == lib.conv3d_fused_pad_workspace_size(1, 2, 5, 5, 5, 1, 16, 1, 1)


def test_dwsep_ex_argument_errors(lib):
    f = lib.dwsep_conv2d_ex
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 5 + [ctypes.c_void_p] * 2 + [ctypes.c_int] + \
        [ctypes.c_void_p] * 2 + [ctypes.c_int, ctypes.c_void_p]
    assert f(FAKE, 1, 4, 5, 5, 4, FAKE, FAKE, 4, None, FAKE, 2, None) == -2   # K = 4
    assert f(FAKE, 1, 4, 5, 5, 9, FAKE, FAKE, 4, None, FAKE, 2, None) == -2   # K = 9
    assert f(FAKE, 1, 16, 8, 8, 7, FAKE, FAKE, 16, None, FAKE, 1, None) == -2  # K = 7 on the TC path
    assert f(FAKE, 1, 24, 8, 8, 5, FAKE, FAKE, 16, None, FAKE, 1, None) == -2  # K = 5 on TC: C not a multiple of 16
    sel = lib.dwsep_conv2d_ex_select_path
    sel.restype = ctypes.c_int
    TC, FMA = 1, 2
    assert sel(16, 64, 512, 512, 5, 128, 0) == TC      # the 5x5 workload: tensor cores
    assert sel(16, 64, 512, 512, 7, 128, 0) == FMA     # 7x7: FMA only
    assert sel(1, 24, 8, 8, 5, 16, 0) == FMA           # C off the 16-channel blocks
    assert sel(1, 16, 8, 8, 5, 16, 2) == FMA           # forced FMA
    assert sel(1, 16, 8, 8, 4, 16, 0) == -2            # K = 4
    assert f(FAKE, 0, 4, 5, 5, 5, FAKE, FAKE, 4, None, FAKE, 0, None) == -1   # N = 0
    assert f(None, 1, 4, 5, 5, 7, FAKE, FAKE, 4, None, FAKE, 0, None) == -1   # NULL x
    assert f(FAKE, 70000, 64, 512, 512, 5, FAKE, FAKE, 4, None, FAKE, 2, None) == -1  # too many elements
