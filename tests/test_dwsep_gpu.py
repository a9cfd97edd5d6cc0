"""GPU parity of dwsep_conv2d (both paths) against the float64 oracle."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from parity import assert_close, sample_indices, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ig3():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_x3x3_gb300 as m
    return m


def paths_for(ig3, N, C, H, W, Cout):
    ps = ["fma"]
    try:
        ig3.dwsep_conv2d_select_path(N, C, H, W, Cout, "tc")
        ps.append("tc")
    except ig3.Ig3Error:
        pass
    return ps


def run(ig3, t, path):
    out = ig3.dwsep_conv2d(to_dev(t["x"]), to_dev(t["w_dw"]), to_dev(t["w_pw"]),
                           to_dev(t["b"]) if "b" in t else None, path=path)
    assert ig3.ig3_last_device_status() == 0
    return out.cpu().numpy()


# (N, C, H, W, Cout, with_bias)
CASES = [
    (2, 16, 9, 70, 32, False),    # ragged tiles in H and W
    (1, 64, 6, 128, 128, True),   # the full-size channel counts, small image, bias
    (1, 32, 5, 36, 48, False),
    (1, 3, 5, 5, 5, True),        # odd channels
    (1, 8, 1, 1, 16, False),      # 1x1 image: only the centre tap sees data
    (2, 8, 2, 4, 16, True),
    (1, 16, 1, 8, 16, False),     # H = 1: both halo rows come from outside the image
    (2, 16, 37, 132, 16, False),  # W = 132: a 4-pixel second segment; strips end mid-image
    (1, 48, 70, 260, 112, True),  # three segments, several strips, Cout 112
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("b" if c[5] else ""))
def test_dwsep_small_all_outputs(ig3, case):
    N, C, H, W, Cout, wb = case
    wl = si.dwsep_workload("t", N, C, H, W, Cout, seed=3000 + N + C + H + W + Cout, with_bias=wb)
    t = wl.generate_all()
    ref = oracle.dwsep(t["x"], t["w_dw"], t["w_pw"], t.get("b"))
    for path in paths_for(ig3, N, C, H, W, Cout):
        assert_close(run(ig3, t, path), ref, f"{case} {path}")


def test_dwsep_full_size_sampled(ig3):
    wl = si.dwsep_conv2d()
    t = wl.generate_all()
    x = to_dev(t["x"]); w_dw = to_dev(t["w_dw"]); w_pw = to_dev(t["w_pw"])
    out = ig3.dwsep_conv2d(x, w_dw, w_pw, None)                     # the benchmark's call
    assert ig3.ig3_last_device_status() == 0
    idx = sample_indices(tuple(out.shape), 8000, seed=5)
    got = out[tuple(torch.from_numpy(idx.T).to(out.device))].cpu().numpy()
    ref = oracle.dwsep_at(t["x"], t["w_dw"], t["w_pw"], None, idx)
    assert_close(got, ref, "dwsep full sampled")
    assert bool(torch.isfinite(out).all())
    del x, w_dw, w_pw, out
    torch.cuda.empty_cache()


def test_dwsep_misaligned_input(ig3):
    """x 4 bytes off a 16-byte boundary: the tensor-core kernel needs 16-byte aligned
    rows, so an explicit request is refused and the automatic choice takes the FMA
    kernel; either way nothing runs on the wrong data."""
    N, C, H, W, Cout = 1, 64, 64, 128, 128      # large enough for the automatic choice to pick TC
    assert ig3.dwsep_conv2d_select_path(N, C, H, W, Cout, "auto") == "tc"
    wl = si.dwsep_workload("t", N, C, H, W, Cout, seed=3100, with_bias=False)
    t = wl.generate_all()
    ref = oracle.dwsep(t["x"], t["w_dw"], t["w_pw"], None)
    buf = torch.empty(t["x"].size + 1, dtype=torch.float32, device="cuda")
    x = buf[1:].view(t["x"].shape)
    x.copy_(torch.from_numpy(t["x"]))
    assert x.data_ptr() % 16 != 0
    w_dw = to_dev(t["w_dw"]); w_pw = to_dev(t["w_pw"])
    with pytest.raises(ig3.Ig3Error):
        ig3.dwsep_conv2d(x, w_dw, w_pw, None, path="tc")
    out = ig3.dwsep_conv2d(x, w_dw, w_pw, None)
    assert ig3.ig3_last_device_status() == 0
    assert_close(out.cpu().numpy(), ref, "misaligned auto")


# ---------------------------------------------------------------- K x K depthwise (FMA path)
# (N, C, H, W, Cout, K): ragged tiles, channel counts off the 8 / 32 blocks, K = 1, 5, 7
# (shapes the tensor-core kernels do not take, so AUTO runs the FMA kernel too).
K_CASES = [
    (1, 5, 9, 70, 33, 5),
    (2, 16, 5, 64, 32, 7),
    (1, 3, 6, 7, 4, 1),
    (1, 8, 2, 3, 8, 7),        # image smaller than the kernel
]


@pytest.mark.parametrize("case", K_CASES, ids=lambda s: "x".join(map(str, s)))
def test_dwsep_k_all_outputs(ig3, case):
    N, C, H, W, Cout, K = case
    wl = si.dwsep_workload("t", N, C, H, W, Cout, seed=3300 + sum(case), with_bias=True, K=K)
    t = wl.generate_all()
    ref = oracle.dwsep_k(t["x"], t["w_dw"], t["w_pw"], t["b"])
    for path in ("auto", "fma"):
        got = ig3.dwsep_conv2d(to_dev(t["x"]), to_dev(t["w_dw"]), to_dev(t["w_pw"]), to_dev(t["b"]), path=path)
        assert ig3.ig3_last_device_status() == 0
        assert_close(got.cpu().numpy(), ref, f"{case} {path}")
    with pytest.raises(ig3.Ig3Error):
        ig3.dwsep_conv2d(to_dev(t["x"]), to_dev(t["w_dw"]), to_dev(t["w_pw"]), None, path="tc")


# ---------------------------------------------------------------- 5x5 depthwise (tensor cores)
# (N, C, H, W, Cout, with_bias): ragged segments and strips, the full channel counts,
# images smaller than the window (H = 1, 2: every halo row from outside the image).
K5_TC_CASES = [
    (2, 16, 9, 68, 32, False),
    (1, 64, 6, 128, 128, True),
    (1, 32, 5, 36, 48, True),
    (1, 16, 1, 8, 16, False),
    (1, 16, 2, 4, 16, True),
    (2, 16, 37, 132, 16, False),
    (1, 48, 70, 260, 112, True),
]


@pytest.mark.parametrize("case", K5_TC_CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("b" if c[5] else ""))
def test_dwsep_k5_tc_all_outputs(ig3, case):
    N, C, H, W, Cout, wb = case
    assert ig3.dwsep_conv2d_ex_select_path(N, C, H, W, 5, Cout, "auto") == "tc"
    wl = si.dwsep_workload("t", N, C, H, W, Cout, seed=3500 + N + C + H + W + Cout, with_bias=wb, K=5)
    t = wl.generate_all()
    ref = oracle.dwsep_k(t["x"], t["w_dw"], t["w_pw"], t.get("b"))
    for path in ("tc", "auto", "fma"):
        assert_close(run(ig3, t, path), ref, f"{case} {path}")


def test_dwsep_k5_misaligned_input(ig3):
    N, C, H, W, Cout = 1, 32, 12, 64, 64
    wl = si.dwsep_workload("t", N, C, H, W, Cout, seed=3590, with_bias=False, K=5)
    t = wl.generate_all()
    ref = oracle.dwsep_k(t["x"], t["w_dw"], t["w_pw"], None)
    buf = torch.empty(t["x"].size + 1, dtype=torch.float32, device="cuda")
    x = buf[1:].view(t["x"].shape)
    x.copy_(torch.from_numpy(t["x"]))
    assert x.data_ptr() % 16 != 0
    w_dw = to_dev(t["w_dw"]); w_pw = to_dev(t["w_pw"])
    with pytest.raises(ig3.Ig3Error):
        ig3.dwsep_conv2d(x, w_dw, w_pw, None, path="tc")
    out = ig3.dwsep_conv2d(x, w_dw, w_pw, None)
    assert ig3.ig3_last_device_status() == 0
    assert_close(out.cpu().numpy(), ref, "K=5 misaligned auto")


def test_dwsep_k5_full_size_sampled(ig3):
    wl = si.dwsep_k5()
    t = wl.generate_all()
    x = to_dev(t["x"]); w_dw = to_dev(t["w_dw"]); w_pw = to_dev(t["w_pw"])
    out = ig3.dwsep_conv2d(x, w_dw, w_pw, None)          # the benchmark's call
    assert ig3.ig3_last_device_status() == 0
    idx = sample_indices(tuple(out.shape), 4000, seed=81)
    rng = np.random.default_rng(82)
    edges = np.stack([rng.integers(0, 16, 400), rng.integers(0, 128, 400),
                      rng.choice([0, 1, 510, 511], 400), rng.choice([0, 1, 510, 511], 400)], 1)
    idx = np.concatenate([idx, edges])
    got = out[tuple(torch.from_numpy(idx.T).to(out.device))].cpu().numpy()
    ref = oracle.dwsep_k_at(t["x"], t["w_dw"], t["w_pw"], None, idx)
    assert_close(got, ref, "dwsep K=5 full sampled")
    del x, w_dw, w_pw, out
    torch.cuda.empty_cache()
