"""conv3d_fused_noalloc: the entry point for callers that cannot allocate device
memory (a runtime that has reserved all device memory up front, a latency-critical
path that cannot take cudaMalloc's device-wide synchronisation, code with no
allocator).  It must give the float64 oracle's results, and the same results as
conv3d_fused with a caller-provided workspace, call after call, while the scratch
comes from the library's own static buffer and holds whatever the previous call
left there.

This file is collected last on purpose, and it must pass both on its own in a
fresh process and after every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from parity import assert_close, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ig3():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_x3x3_gb300 as m
    return m


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def oracle_ref(t, epi, divisor=2.0):
    """The float64 oracle's result for one case."""
    if epi == "pool_reduce":
        return oracle.conv3d_pool_reduce(t["x"], t["w"], t["b"], divisor, 2, t["bias2"])
    y = oracle.conv3d(t["x"], t["w"], t["b"])
    return oracle.tanh_mish(y) if epi == "tanh_mish" else y


def noalloc_call(ig3, x, w, b, epi, params, out, path):
    """One call of the new entry point straight through the C ABI."""
    N, Cin, D, H, W = x.shape
    Cout = w.shape[0]
    pr = None
    if params is not None:
        pr = ig3._EpiParams(float(params["divisor"]), int(params["pool"]), params["bias2"].data_ptr())
    stream = torch.cuda.current_stream().cuda_stream
    return ig3.lib.conv3d_fused_noalloc(_ptr(x), N, Cin, D, H, W, _ptr(w), Cout, _ptr(b), ig3.EPILOGUES[epi],
                                        None if pr is None else ctypes.byref(pr), _ptr(out), ig3.PATHS[path],
                                        ctypes.c_void_p(stream))


CASES = [
    # (N, Cin, D, H, W, Cout, epilogue, path)
    (2, 16, 5, 10, 64, 32, "tanh_mish", "tc"),    # scratch: split weights
    (2, 8, 6, 10, 64, 16, "pool_reduce", "tc"),   # scratch: split weights + partial sums
    (2, 8, 6, 10, 64, 16, "pool_reduce", "fma"),  # scratch: partial sums
    (1, 4, 5, 6, 7, 8, "tanh_mish", "auto"),      # needs no scratch at all
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + f"-{c[6]}-{c[7]}")
def test_noalloc_matches_conv3d_fused_twice(ig3, case):
    N, Cin, D, H, W, Cout, epi, path = case
    wl = si.conv3d_workload("noalloc", N, Cin, D, H, W, Cout, seed=4000 + sum(case[:6]), epilogue=epi,
                            bias2=(epi == "pool_reduce"))
    t = wl.generate_all()
    x, w, b = to_dev(t["x"]), to_dev(t["w"]), to_dev(t["b"])
    params = None
    if epi == "pool_reduce":
        params = {"divisor": 2.0, "pool": 2, "bias2": to_dev(t["bias2"])}
    need = ig3.conv3d_fused_workspace_size(N, Cin, D, H, W, Cout, epi, path)
    assert need <= ig3.NOALLOC_SCRATCH_BYTES
    ref = oracle_ref(t, epi)
    via_workspace = ig3.conv3d_fused(x, w, b, epilogue=epi, params=params, path=path).cpu().numpy()
    assert_close(via_workspace, ref, f"conv3d_fused {case}")
    for call in range(2):
        out = torch.full(ref.shape, float("nan"), device="cuda")
        st = noalloc_call(ig3, x, w, b, epi, params, out, path)
        assert st == 0, ig3.ig3_last_error()
        torch.cuda.synchronize()
        assert ig3.ig3_last_device_status() == 0
        got = out.cpu().numpy()
        assert_close(got, ref, f"noalloc call {call + 1} {case} vs the oracle")
        assert_close(got, via_workspace, f"noalloc call {call + 1} {case} vs conv3d_fused")


def test_noalloc_after_a_larger_call(ig3):
    # A call with a large weight blob fills the shared scratch; a following smaller
    # call must not depend on what is left there (its partial sums sit where the
    # earlier blob was).
    def case(N, Cin, D, H, W, seed):
        wl = si.conv3d_workload("noalloc_seq", N, Cin, D, H, W, 16, seed=seed, epilogue="pool_reduce", bias2=True)
        t = wl.generate_all()
        dev = {k: to_dev(v) for k, v in t.items()}
        params = {"divisor": 2.0, "pool": 2, "bias2": dev["bias2"]}
        return t, dev, params
    big_t, big, big_p = case(2, 40, 6, 10, 64, 4201)
    small_t, small, small_p = case(3, 8, 6, 12, 64, 4202)
    assert ig3.conv3d_fused_workspace_size(2, 40, 6, 10, 64, 16, "pool_reduce", "tc") > \
        ig3.conv3d_fused_workspace_size(3, 8, 6, 12, 64, 16, "pool_reduce", "tc")
    for t, dev, params, n in ((big_t, big, big_p, 2), (small_t, small, small_p, 3), (small_t, small, small_p, 3)):
        out = torch.full((n,), float("nan"), device="cuda")
        st = noalloc_call(ig3, dev["x"], dev["w"], dev["b"], "pool_reduce", params, out, "tc")
        assert st == 0, ig3.ig3_last_error()
        torch.cuda.synchronize()
        assert ig3.ig3_last_device_status() == 0
        assert_close(out.cpu().numpy(), oracle_ref(t, "pool_reduce"), f"noalloc sequence N={n}")


def test_noalloc_rejects_shapes_beyond_its_buffer(ig3):
    # Cin = 256, Cout = 128 on tensor cores needs about 7 MB of split weights.
    x = torch.zeros(1, 256, 3, 3, 64, device="cuda")
    w = torch.zeros(128, 256, 3, 3, 3, device="cuda")
    out = torch.full((1, 128, 1, 1, 62), 7.0, device="cuda")
    assert ig3.conv3d_fused_workspace_size(1, 256, 3, 3, 64, 128, "none", "tc") > ig3.NOALLOC_SCRATCH_BYTES
    st = noalloc_call(ig3, x, w, None, "none", None, out, "tc")
    assert st == -5  # IG3_ERR_WORKSPACE
    assert "scratch" in ig3.ig3_last_error()
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())  # nothing was launched
    with pytest.raises(ig3.Ig3Error):
        ig3.conv3d_fused_noalloc(x, w, None, epilogue="none", out=out, path="tc")


def test_noalloc_python_binding(ig3):
    wl = si.conv3d_workload("noalloc_py", 1, 8, 4, 6, 64, 16, seed=4100, epilogue="tanh_mish")
    t = wl.generate_all()
    x, w, b = to_dev(t["x"]), to_dev(t["w"]), to_dev(t["b"])
    ref = oracle_ref(t, "tanh_mish")
    got = ig3.conv3d_fused_noalloc(x, w, b, path="tc").cpu().numpy()
    assert ig3.ig3_last_device_status() == 0
    assert_close(got, ref, "noalloc binding")
    assert np.isfinite(got).all()
