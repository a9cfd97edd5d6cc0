"""GPU parity of conv3d_fused (both paths) against the float64 oracle.

Small cases are compared element by element on every output; the full-size
workloads (in the launch configuration the benchmark times) are compared on
sampled outputs the oracle computes one by one.
"""
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


def tc_supported(ig3, N, Cin, D, H, W, Cout, epi):
    try:
        ig3.conv3d_fused_select_path(N, Cin, D, H, W, Cout, epi, "tc")
        return True
    except ig3.Ig3Error:
        return False


def run_conv(ig3, t, epi, path, params=None):
    x = to_dev(t["x"]); w = to_dev(t["w"])
    b = to_dev(t["b"]) if "b" in t else None
    dev_params = None
    if epi == "pool_reduce":
        dev_params = dict(params or {})
        dev_params["bias2"] = to_dev(t["bias2"])
    out = ig3.conv3d_fused(x, w, b, epilogue=epi, params=dev_params, path=path)
    assert ig3.ig3_last_device_status() == 0
    return out.cpu().numpy()


def paths_for(ig3, shape, epi):
    N, Cin, D, H, W, Cout = shape
    ps = ["fma"]
    if tc_supported(ig3, N, Cin, D, H, W, Cout, epi):
        ps.append("tc")
    return ps


# (N, Cin, D, H, W, Cout): several tiles of both kernels and ragged tails in every dim.
SMALL_CASES = [
    (2, 32, 6, 20, 70, 64),   # ragged columns and rows for both tilings
    (1, 8, 5, 11, 64, 16),    # W = 64 (two input rows per 128-position tile)
    (2, 16, 4, 9, 8, 16),     # narrow rows (W = 8)
    (1, 16, 4, 6, 64, 128),   # Cout = 128
    (1, 24, 3, 7, 33, 48),    # Cin not a multiple of 8, Cout = 48
    (1, 40, 5, 10, 32, 32),   # Cout = 32: hi and lo products in separate accumulator columns
    (1, 5, 4, 11, 13, 80),    # Cout = 80: the widest three-plane window (N = 240)
    (1, 12, 5, 8, 20, 96),    # Cout = 96: one MMA per kd over a ring of five slots
    (1, 8, 6, 9, 16, 112),    # Cout = 112: one MMA per kd, four slots
    (2, 72, 4, 6, 24, 64),    # Cin = 72: several channel chunks of streamed weights
    (1, 8, 5, 6, 4, 16),      # Cout = 16, kw inside the MMA (window over kd and kw): W = 4
    (2, 8, 6, 12, 32, 16),    #   W = 32: rows end at quadrant ends
    (1, 8, 6, 12, 128, 16),   #   W = 128: one row per tile, three quadrant crossings
    (2, 8, 10, 64, 64, 16),   #   two position tiles per unit
    (1, 40, 5, 6, 64, 16),    #   five K-steps of resident weights
    (1, 136, 5, 6, 64, 16),   #   streamed weights
    (1, 8, 5, 9, 20, 16),     # Cout = 16 with W not dividing 128: hi and lo columns instead
    (1, 12, 9, 7, 64, 16),    # Cout = 16, A in tensor memory: a half-empty second K-step
    (2, 3, 7, 5, 32, 16),     #   three input channels
    (1, 24, 12, 6, 16, 16),   #   three channel chunks per plane
    (3, 8, 20, 10, 64, 16),   #   many planes per unit: the slot ring wraps inside units
    (1, 32, 12, 6, 128, 16),  #   two chunks of two K-steps, W = 128
    (2, 16, 6, 5, 12, 16),    #   H*W % 4 == 0 but W not dividing 128: the other kernel
    (1, 8, 5, 7, 6, 16),      #   H*W % 4 != 0: the other kernel
    (2, 3, 5, 7, 9, 5),       # odd channel counts
    (1, 1, 3, 3, 3, 1),       # smallest valid input: one output
]


@pytest.mark.parametrize("shape", SMALL_CASES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("epi", ["tanh_mish", "none"])
def test_conv3d_small_all_outputs(ig3, shape, epi):
    N, Cin, D, H, W, Cout = shape
    wl = si.conv3d_workload("t", N, Cin, D, H, W, Cout, seed=1000 + sum(shape), epilogue=epi)
    t = wl.generate_all()
    y = oracle.conv3d(t["x"], t["w"], t["b"])
    ref = oracle.tanh_mish(y) if epi == "tanh_mish" else y
    for path in paths_for(ig3, shape, epi):
        got = run_conv(ig3, t, epi, path)
        assert_close(got, ref, f"{shape} {epi} {path}")


def test_tiny_workload_all_outputs(ig3):
    wl = si.tiny_conv3d()
    t = wl.generate_all()
    ref = oracle.conv3d_tanh_mish(t["x"], t["w"], t["b"])
    for path in paths_for(ig3, tuple(wl.dims.values()), "tanh_mish") + ["auto"]:
        assert_close(run_conv(ig3, t, "tanh_mish", path), ref, f"tiny {path}")


def test_conv3d_without_bias(ig3):
    wl = si.conv3d_workload("t", 1, 16, 4, 8, 64, 32, seed=77, epilogue="tanh_mish", with_bias=False)
    t = wl.generate_all()
    ref = oracle.conv3d_tanh_mish(t["x"], t["w"], None)
    for path in paths_for(ig3, (1, 16, 4, 8, 64, 32), "tanh_mish"):
        assert_close(run_conv(ig3, t, "tanh_mish", path), ref, f"no bias {path}")


@pytest.mark.parametrize("shape", [(1, 8, 4, 6, 64, 16), (1, 8, 4, 6, 64, 64), (1, 8, 4, 6, 128, 16)],
                         ids=["cout16_a_in_tmem", "cout64_kd_window", "cout16_kd_kw_window"])
def test_activation_over_wide_range(ig3, shape):
    # Large weights drive conv outputs across [-60, 60]: exercises both branches
    # of the activation and its saturation, in each tensor-core epilogue.
    wl = si.conv3d_workload("t", *shape, seed=78, epilogue="tanh_mish", wb_bound=2.5,
                            x_dist=("uniform", -3.0, 3.0))
    t = wl.generate_all()
    y = oracle.conv3d(t["x"], t["w"], t["b"])
    assert y.min() < -20 and y.max() > 20
    ref = oracle.tanh_mish(y)
    for path in paths_for(ig3, shape, "tanh_mish"):
        assert_close(run_conv(ig3, t, "tanh_mish", path), ref, f"wide range {path}")


# ---------------------------------------------------------------- full-size, sampled
FULL = {
    "conv3d_tanh_mish": si.conv3d_tanh_mish,
    "sweep16": lambda: si.conv3d_sweep(16),
    "sweep64": lambda: si.conv3d_sweep(64),
    "sweep128": lambda: si.conv3d_sweep(128),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled(ig3, name):
    wl = FULL[name]()
    t = wl.generate_all()
    d = wl.dims
    x = to_dev(t["x"]); w = to_dev(t["w"]); b = to_dev(t["b"])
    out = ig3.conv3d_fused(x, w, b, epilogue="tanh_mish")          # the benchmark's call
    assert ig3.ig3_last_device_status() == 0
    idx = sample_indices(tuple(out.shape), 6000, seed=len(name))
    got = out[tuple(torch.from_numpy(idx.T).to(out.device))].cpu().numpy()
    ref = oracle.tanh_mish(oracle.conv3d_at(t["x"], t["w"], t["b"], idx))
    assert_close(got, ref, f"{name} sampled")
    # Every output is finite and inside the range of tanh.
    assert bool(torch.isfinite(out).all()) and float(out.abs().max()) <= 1.0
    del x, w, b, out
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- pool-reduce
POOL_CASES = [
    (3, 8, 6, 10, 64, 16),    # W = 64: two rows per tensor-core tile
    (2, 8, 6, 8, 8, 16),      # W = 8
    (2, 4, 7, 9, 13, 16),     # odd conv-output dims: floor mode drops a plane, row, column
    (1, 5, 4, 4, 4, 3),       # smallest pooled grid (1x1x1), odd channels
    (2, 16, 5, 12, 32, 32),   # W = 32, odd conv-output depth
    (2, 8, 6, 10, 16, 16),    # W = 16: h-pair by lane shuffle
    (2, 8, 6, 10, 32, 16),    # W = 32
    (1, 8, 6, 12, 4, 16),     # W = 4
    (2, 8, 8, 64, 64, 16),    # two position tiles per unit
    (2, 3, 7, 5, 32, 16),     # odd conv-output depth, three input channels
    (4, 8, 33, 10, 64, 16),   # 31 conv-output planes: several plane splits
    (1, 12, 9, 7, 16, 16),    # a half-empty second K-step, odd depth
    (3, 24, 6, 6, 8, 16),     # three channel chunks
]


@pytest.mark.parametrize("shape", POOL_CASES, ids=lambda s: "x".join(map(str, s)))
def test_pool_reduce_small(ig3, shape):
    N, Cin, D, H, W, Cout = shape
    wl = si.conv3d_workload("t", N, Cin, D, H, W, Cout, seed=2000 + sum(shape), epilogue="pool_reduce",
                            bias2=True)
    t = wl.generate_all()
    for div in (2.0, -1.5):
        ref = oracle.conv3d_pool_reduce(t["x"], t["w"], t["b"], div, 2, t["bias2"])
        for path in paths_for(ig3, shape, "pool_reduce"):
            got = run_conv(ig3, t, "pool_reduce", path, params={"divisor": div, "pool": 2})
            assert_close(got, ref, f"{shape} div={div} {path}")


# One shape per streamed-weight kernel variant (KDM, HL, T, KSS, taps per weight stage),
# each the cheapest multi-tile shape the planner maps to it; tests/planner_check.cu
# asserts the same mapping on the CPU.  Every output against the oracle.
STAGE_CASES = [
    # (N, Cin, D, H, W, Cout), epilogue
    ((1, 9, 5, 4, 280, 96), "tanh_mish"),    # KDM 1, 1 K-step chunks, 1 tap per stage
    ((1, 9, 5, 4, 184, 96), "tanh_mish"),    # KDM 1, 1 K-step chunks, 2 taps
    ((1, 17, 5, 48, 8, 96), "tanh_mish"),    # KDM 1, 1 K-step chunks, 3 taps
    ((1, 17, 5, 48, 8, 96), "pool_reduce"),
    ((8, 9, 6, 4, 288, 96), "none"),         # KDM 1, 2 K-step chunks, 1 tap
    ((1, 9, 5, 4, 192, 128), "tanh_mish"),   # KDM 1, 2 K-step chunks, 2 taps
    ((1, 9, 5, 48, 8, 96), "pool_reduce"),   # KDM 1, 2 K-step chunks, 3 taps
    ((1, 9, 5, 4, 240, 48), "tanh_mish"),    # KDM 3, one tile, 1 tap
    ((1, 9, 5, 4, 168, 48), "tanh_mish"),    # KDM 3, one tile, 2 taps
    ((1, 9, 5, 48, 8, 80), "pool_reduce"),
    ((1, 9, 5, 4, 152, 48), "none"),         # KDM 3, one tile, 3 taps
    ((1, 9, 5, 48, 8, 64), "pool_reduce"),
    ((4, 9, 12, 4, 200, 48), "tanh_mish"),   # KDM 3, two tiles, 1 tap
    ((8, 9, 5, 48, 32, 80), "pool_reduce"),
    ((4, 9, 6, 9, 168, 48), "tanh_mish"),    # KDM 3, two tiles, 2 taps
    ((8, 9, 5, 48, 32, 64), "pool_reduce"),
    ((4, 9, 5, 33, 96, 48), "tanh_mish"),    # KDM 3, two tiles, 3 taps
    ((8, 9, 5, 48, 32, 48), "pool_reduce"),
    ((1, 9, 5, 4, 288, 16), "tanh_mish"),    # KDM 3 hi/lo columns, one tile, 1 tap
    ((1, 9, 5, 4, 248, 16), "none"),         # KDM 3 hi/lo columns, one tile, 2 taps
    ((1, 9, 5, 48, 8, 32), "tanh_mish"),     # KDM 3 hi/lo columns, one tile, 3 taps
    ((1, 9, 5, 48, 8, 32), "pool_reduce"),
    ((4, 17, 12, 4, 224, 16), "tanh_mish"),  # KDM 3 hi/lo columns, two tiles, 1 tap
    ((4, 17, 12, 4, 200, 16), "tanh_mish"),  # KDM 3 hi/lo columns, two tiles, 2 taps
    ((8, 9, 5, 48, 32, 32), "pool_reduce"),
    ((8, 17, 5, 9, 168, 16), "tanh_mish"),   # KDM 3 hi/lo columns, two tiles, 3 taps
    ((1, 57, 5, 6, 128, 16), "tanh_mish"),   # KDM 9 (kd x kw window), one tile, streamed
    ((4, 57, 12, 6, 128, 16), "tanh_mish"),  # KDM 9, two tiles, streamed
]


@pytest.mark.parametrize("case", STAGE_CASES, ids=lambda c: "x".join(map(str, c[0])) + "-" + c[1])
def test_conv3d_weight_stage_variants_all_outputs(ig3, case):
    shape, epi = case
    N, Cin, D, H, W, Cout = shape
    assert tc_supported(ig3, N, Cin, D, H, W, Cout, epi)
    wl = si.conv3d_workload("t", N, Cin, D, H, W, Cout, seed=3000 + sum(shape), epilogue=epi,
                            bias2=(epi == "pool_reduce"))
    t = wl.generate_all()
    if epi == "pool_reduce":
        ref = oracle.conv3d_pool_reduce(t["x"], t["w"], t["b"], 2.0, 2, t["bias2"])
        got = run_conv(ig3, t, epi, "tc", params={"divisor": 2.0, "pool": 2})
    else:
        y = oracle.conv3d(t["x"], t["w"], t["b"])
        ref = oracle.tanh_mish(y) if epi == "tanh_mish" else y
        got = run_conv(ig3, t, epi, "tc")
    assert_close(got, ref, f"{shape} {epi}")


def test_pool_reduce_full_size_sampled_and_deterministic(ig3):
    wl = si.conv3d_pool_reduce()
    t = wl.generate_all()
    x = to_dev(t["x"]); w = to_dev(t["w"]); b = to_dev(t["b"]); bias2 = to_dev(t["bias2"])
    params = {"divisor": 2.0, "pool": 2, "bias2": bias2}
    out1 = ig3.conv3d_fused(x, w, b, epilogue="pool_reduce", params=params).cpu().numpy()
    out2 = ig3.conv3d_fused(x, w, b, epilogue="pool_reduce", params=params).cpu().numpy()
    assert ig3.ig3_last_device_status() == 0
    assert out1.shape == (128,)
    assert np.array_equal(out1, out2), "pool-reduce is not deterministic"
    # Every one of the 128 outputs against the oracle (47.6 GFLOP of float64 work).
    ref = oracle.conv3d_pool_reduce(t["x"], t["w"], t["b"], 2.0, 2, t["bias2"])
    assert_close(out1, ref, "pool-reduce full size, all outputs")


def test_headline_full_size_every_element(ig3):
    # The conv3d + tanh(mish) workload in the benchmark's launch configuration,
    # compared with the oracle on every one of its 118,087,680 outputs (one batch
    # item of the oracle at a time).
    wl = si.conv3d_tanh_mish()
    t = wl.generate_all()
    x = to_dev(t["x"]); w = to_dev(t["w"]); b = to_dev(t["b"])
    out = ig3.conv3d_fused(x, w, b, epilogue="tanh_mish")
    assert ig3.ig3_last_device_status() == 0
    got = out.cpu().numpy()
    del x, w, b, out
    torch.cuda.empty_cache()
    for n in range(got.shape[0]):
        ref = oracle.conv3d_tanh_mish(t["x"][n:n + 1], t["w"], t["b"])
        assert_close(got[n:n + 1], ref, f"conv3d + tanh(mish) full size, batch item {n}")


def test_cout16_misaligned_input(ig3):
    # x one float past a 16-byte boundary: the tensor-core path still runs (the kernel
    # that copies 16-byte channel rows needs an aligned x, the other one does not).
    wl = si.conv3d_workload("t", 1, 8, 5, 10, 64, 16, seed=93, epilogue="tanh_mish")
    t = wl.generate_all()
    ref = oracle.conv3d_tanh_mish(t["x"], t["w"], t["b"])
    xs = torch.zeros(t["x"].size + 1, device="cuda")
    xs[1:] = to_dev(t["x"]).reshape(-1)
    x = xs[1:].view(t["x"].shape)
    assert x.data_ptr() % 16 != 0
    out = ig3.conv3d_fused(x, to_dev(t["w"]), to_dev(t["b"]), epilogue="tanh_mish", path="tc")
    assert ig3.ig3_last_device_status() == 0
    assert_close(out.cpu().numpy(), ref, "misaligned x, Cout 16, tc")


# ---------------------------------------------------------------- edges of the boundary
def test_output_canaries_untouched(ig3):
    wl = si.conv3d_workload("t", 1, 8, 5, 9, 64, 16, seed=91, epilogue="tanh_mish")
    t = wl.generate_all()
    x = to_dev(t["x"]); w = to_dev(t["w"]); b = to_dev(t["b"])
    n_out = 1 * 16 * 3 * 7 * 62
    for path in paths_for(ig3, (1, 8, 5, 9, 64, 16), "tanh_mish"):
        buf = torch.full((n_out + 2048,), 12345.0, device="cuda")
        out = buf[1024:1024 + n_out].view(1, 16, 3, 7, 62)
        ig3.conv3d_fused(x, w, b, epilogue="tanh_mish", out=out, path=path)
        torch.cuda.synchronize()
        assert bool((buf[:1024] == 12345.0).all()) and bool((buf[1024 + n_out:] == 12345.0).all()), path


def test_errors_are_reported_not_raised_on_device(ig3):
    x = torch.zeros(1, 2, 3, 3, 3, device="cuda")
    w = torch.zeros(2, 2, 3, 3, 3, device="cuda")
    with pytest.raises(ig3.Ig3Error) as e:
        ig3.conv3d_fused(x, w, None, epilogue="pool_reduce", params={"bias2": torch.zeros(2, device="cuda")})
    assert e.value.status == -2  # 1x1x1 conv output: the pooled grid is empty
    with pytest.raises(ig3.Ig3Error) as e:
        ig3.conv3d_fused(x, w, None, epilogue="tanh_mish", path="tc")
    assert e.value.status == -2  # Cout = 2 is not a tensor-core shape
    torch.cuda.synchronize()
    assert ig3.ig3_last_device_status() == 0


@pytest.mark.parametrize("shape,epi", [((1, 8, 6, 10, 64, 16), "pool_reduce"), ((1, 32, 5, 8, 64, 64), "tanh_mish"),
                                       ((1, 16, 5, 9, 16, 32), "tanh_mish")],
                         ids=["pool-resident", "streamed", "split-columns"])
def test_conv3d_misaligned_input(ig3, shape, epi):
    """x 4 bytes off a 16-byte boundary: the convert falls back from 16-byte loads and
    from the bulk-copy loader to scalar loads; results must not change."""
    N, Cin, D, H, W, Cout = shape
    wl = si.conv3d_workload("t", N, Cin, D, H, W, Cout, seed=5000 + sum(shape), epilogue=epi,
                            bias2=(epi == "pool_reduce"))
    t = wl.generate_all()
    params = {"divisor": 2.0, "pool": 2} if epi == "pool_reduce" else None
    if epi == "pool_reduce":
        ref = oracle.conv3d_pool_reduce(t["x"], t["w"], t["b"], 2.0, 2, t["bias2"])
    else:
        ref = oracle.tanh_mish(oracle.conv3d(t["x"], t["w"], t["b"]))
    buf = torch.empty(t["x"].size + 1, dtype=torch.float32, device="cuda")
    x = buf[1:].view(t["x"].shape)
    x.copy_(torch.from_numpy(t["x"]))
    assert x.data_ptr() % 16 != 0
    w = to_dev(t["w"]); b = to_dev(t["b"])
    dev_params = None
    if params is not None:
        dev_params = dict(params)
        dev_params["bias2"] = to_dev(t["bias2"])
    for path in paths_for(ig3, shape, epi):
        out = ig3.conv3d_fused(x, w, b, epilogue=epi, params=dev_params, path=path)
        assert ig3.ig3_last_device_status() == 0
        assert_close(out.cpu().numpy(), ref, f"misaligned {shape} {epi} {path}")


# ---------------------------------------------------------------- zero padding
def tc_supported_pad(ig3, shape, pad, epi):
    N, Cin, D, H, W, Cout = shape
    return tc_supported(ig3, N, Cin, D + 2 * pad, H + 2 * pad, W + 2 * pad, Cout, epi)


# (N, Cin, D, H, W, Cout, pad): the tensor-core variants the padded shapes select
# (kd x kw window, split columns, kd window), pad 2, and shapes only FMA takes.
PAD_CASES = [
    (1, 8, 4, 9, 62, 16, 1),    # padded W = 64: Cout 16 kd x kw window
    (2, 16, 5, 7, 30, 32, 1),   # padded W = 32: split hi/lo columns
    (1, 24, 3, 5, 20, 64, 1),   # kd window, Cin not a multiple of 16
    (1, 4, 3, 3, 3, 16, 2),     # pad 2, a 3x3x3 input
    (1, 3, 2, 3, 4, 5, 1),      # D = 2 input (valid conv impossible), odd channels: FMA
    (2, 5, 1, 1, 1, 16, 1),     # single voxel: one output per channel
    # the border filled on chip: W % 4 == 0 gives aligned 16-byte loads over a virtual
    # row pitch of W + 4 (pad <= 4), other widths scalar loads over W + 2*pad
    (2, 32, 6, 10, 64, 64, 1),  # pitch 68, kd window (the padded workload's variant)
    (1, 16, 5, 7, 60, 16, 2),   # pitch 64: Cout 16 kd x kw window
    (1, 8, 4, 6, 32, 96, 3),    # pitch 36, one MMA per kd
    (1, 8, 5, 5, 16, 32, 4),    # pitch 20, pad 4: the whole left border is the virtual row's first quad
    (1, 8, 4, 5, 8, 48, 5),     # pad 5: scalar loads over pitch 18
    (2, 12, 5, 6, 13, 64, 1),   # W % 4 != 0: scalar loads over pitch 15
]


@pytest.mark.parametrize("case", PAD_CASES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("epi", ["tanh_mish", "none"])
def test_conv3d_pad_small_all_outputs(ig3, case, epi):
    *shape, pad = case
    N, Cin, D, H, W, Cout = shape
    wl = si.conv3d_workload("t", N, Cin, D, H, W, Cout, seed=3000 + sum(case), epilogue=epi, pad=pad)
    t = wl.generate_all()
    y = oracle.conv3d_pad(t["x"], t["w"], t["b"], pad)
    ref = oracle.tanh_mish(y) if epi == "tanh_mish" else y
    paths = ["fma"] + (["tc"] if tc_supported_pad(ig3, tuple(shape), pad, epi) else [])
    for path in paths:
        x = to_dev(t["x"]); w = to_dev(t["w"]); b = to_dev(t["b"])
        got = ig3.conv3d_fused(x, w, b, epilogue=epi, path=path, pad=pad)
        assert ig3.ig3_last_device_status() == 0
        assert tuple(got.shape) == ref.shape
        assert_close(got.cpu().numpy(), ref, f"{case} {epi} {path}")


@pytest.mark.parametrize("case", [(2, 8, 6, 8, 62, 16, 1), (1, 4, 5, 5, 5, 16, 1), (2, 8, 7, 6, 28, 32, 2),
                                  (1, 8, 6, 9, 30, 16, 1)],
                         ids=lambda s: "x".join(map(str, s)))
def test_conv3d_pad_pool_reduce(ig3, case):
    *shape, pad = case
    N, Cin, D, H, W, Cout = shape
    wl = si.conv3d_workload("t", N, Cin, D, H, W, Cout, seed=3100 + sum(case), epilogue="pool_reduce",
                            bias2=True, pad=pad)
    t = wl.generate_all()
    ref = oracle.pool_reduce(oracle.conv3d_pad(t["x"], t["w"], t["b"], pad), 2.0, 2, t["bias2"])
    paths = ["fma"] + (["tc"] if tc_supported_pad(ig3, tuple(shape), pad, "pool_reduce") else [])
    for path in paths:
        got = ig3.conv3d_fused(to_dev(t["x"]), to_dev(t["w"]), to_dev(t["b"]), epilogue="pool_reduce",
                               params={"divisor": 2.0, "pool": 2, "bias2": to_dev(t["bias2"])}, path=path, pad=pad)
        assert ig3.ig3_last_device_status() == 0
        assert_close(got.cpu().numpy(), ref, f"{case} pool {path}")


def test_conv3d_pad_misaligned_input(ig3):
    # x one float past a 16-byte boundary: the padded tensor-core path loads it with
    # scalar loads over a virtual pitch of W + 2*pad.
    wl = si.conv3d_workload("t", 1, 16, 5, 8, 64, 64, seed=3190, epilogue="tanh_mish", pad=1)
    t = wl.generate_all()
    ref = oracle.tanh_mish(oracle.conv3d_pad(t["x"], t["w"], t["b"], 1))
    xs = torch.zeros(t["x"].size + 1, device="cuda")
    xs[1:] = to_dev(t["x"]).reshape(-1)
    x = xs[1:].view(t["x"].shape)
    assert x.data_ptr() % 16 != 0
    got = ig3.conv3d_fused(x, to_dev(t["w"]), to_dev(t["b"]), epilogue="tanh_mish", path="tc", pad=1)
    assert ig3.ig3_last_device_status() == 0
    assert_close(got.cpu().numpy(), ref, "padded, misaligned x, tc")


def test_conv3d_pad_full_size_sampled(ig3):
    wl = si.conv3d_same_tanh_mish()
    t = wl.generate_all()
    x = to_dev(t["x"]); w = to_dev(t["w"]); b = to_dev(t["b"])
    out = ig3.conv3d_fused(x, w, b, epilogue="tanh_mish", pad=wl.pad)   # the benchmark's call
    assert ig3.ig3_last_device_status() == 0
    assert tuple(out.shape) == (16, 64, 32, 64, 64)
    idx = sample_indices(tuple(out.shape), 6000, seed=61)
    # Include the faces, edges and corners, where the zero border is read.
    rng = np.random.default_rng(62)
    faces = np.stack([rng.integers(0, 16, 600), rng.integers(0, 64, 600),
                      rng.choice([0, 31], 600), rng.choice([0, 63], 600), rng.integers(0, 64, 600)], 1)
    idx = np.concatenate([idx, faces])
    got = out[tuple(torch.from_numpy(idx.T).to(out.device))].cpu().numpy()
    ref = oracle.tanh_mish(oracle.conv3d_pad_at(t["x"], t["w"], t["b"], wl.pad, idx))
    assert_close(got, ref, "conv3d pad 1 full size sampled")
    del x, w, b, out
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- stride 2 (FMA path)
# (N, Cin, D, H, W, Cout, pad): ragged tiles in every dim, Cout not a multiple of the
# 16-channel block, odd and even input sizes, pad 0..2 (shapes the tensor-core kernel
# does not take, so AUTO runs the FMA kernel too).
STRIDE2_CASES = [
    (1, 3, 7, 9, 11, 5, 0),
    (2, 4, 8, 20, 70, 16, 1),
    (1, 2, 5, 6, 5, 33, 1),
    (1, 5, 4, 4, 4, 8, 2),
    (1, 1, 3, 3, 3, 1, 0),      # one output
]


@pytest.mark.parametrize("case", STRIDE2_CASES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("epi", ["tanh_mish", "none"])
def test_conv3d_stride2_all_outputs(ig3, case, epi):
    *shape, pad = case
    N, Cin, D, H, W, Cout = shape
    wl = si.conv3d_workload("t", N, Cin, D, H, W, Cout, seed=3200 + sum(case), epilogue=epi, pad=pad)
    t = wl.generate_all()
    y = oracle.conv3d_ex(t["x"], t["w"], t["b"], pad, 2)
    ref = oracle.tanh_mish(y) if epi == "tanh_mish" else y
    for path in ("auto", "fma"):
        got = ig3.conv3d_fused(to_dev(t["x"]), to_dev(t["w"]), to_dev(t["b"]), epilogue=epi, path=path,
                               pad=pad, stride=2)
        assert ig3.ig3_last_device_status() == 0
        assert tuple(got.shape) == ref.shape
        assert_close(got.cpu().numpy(), ref, f"{case} {epi} {path}")
    got = ig3.conv3d_fused(to_dev(t["x"]), to_dev(t["w"]), None, epilogue=epi, pad=pad, stride=2)
    y0 = oracle.conv3d_ex(t["x"], t["w"], None, pad, 2)
    assert_close(got.cpu().numpy(), oracle.tanh_mish(y0) if epi == "tanh_mish" else y0, f"{case} no bias")


# ---------------------------------------------------------------- stride 2 (tensor cores)
# (N, Cin, D, H, W, Cout, pad): both A-stage shapes of the gathering kernel (three
# kernel rows for Cout <= 112, one row for 128), ragged position tiles, Cin not a
# multiple of 8, pad 0..5, and an output plane whose whole window lies in the padding
# (bias only).
STRIDE2_TC_CASES = [
    (1, 3, 7, 9, 12, 16, 0),
    (2, 8, 8, 20, 68, 32, 1),
    (1, 5, 5, 6, 8, 48, 2),
    (1, 12, 9, 33, 36, 64, 1),
    (1, 8, 5, 8, 16, 96, 1),
    (1, 40, 6, 12, 36, 128, 1),
    (1, 8, 4, 4, 4, 16, 3),
    (2, 24, 16, 64, 64, 64, 1),
    (1, 8, 5, 6, 8, 16, 5),       # pad 5: the staged box starts 8 columns left of x
    (1, 16, 7, 10, 24, 112, 2),   # Cout 112: the widest three-row A stages
]


@pytest.mark.parametrize("case", STRIDE2_TC_CASES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("epi", ["tanh_mish", "none"])
def test_conv3d_stride2_tc_all_outputs(ig3, case, epi):
    *shape, pad = case
    N, Cin, D, H, W, Cout = shape
    e = 1 if epi == "tanh_mish" else 0
    assert ig3.lib.conv3d_fused_ex_workspace_size(N, Cin, D, H, W, pad, 2, Cout, e, 1) > 0  # the TC path applies
    wl = si.conv3d_workload("t", N, Cin, D, H, W, Cout, seed=3300 + sum(case), epilogue=epi, pad=pad)
    t = wl.generate_all()
    y = oracle.conv3d_ex(t["x"], t["w"], t["b"], pad, 2)
    ref = oracle.tanh_mish(y) if epi == "tanh_mish" else y
    for path in ("tc", "auto"):
        got = ig3.conv3d_fused(to_dev(t["x"]), to_dev(t["w"]), to_dev(t["b"]), epilogue=epi, path=path,
                               pad=pad, stride=2)
        assert ig3.ig3_last_device_status() == 0
        assert tuple(got.shape) == ref.shape
        assert_close(got.cpu().numpy(), ref, f"{case} {epi} {path}")
    got = ig3.conv3d_fused(to_dev(t["x"]), to_dev(t["w"]), None, epilogue=epi, path="tc", pad=pad, stride=2)
    y0 = oracle.conv3d_ex(t["x"], t["w"], None, pad, 2)
    assert_close(got.cpu().numpy(), oracle.tanh_mish(y0) if epi == "tanh_mish" else y0, f"{case} no bias")


def test_conv3d_stride2_tc_misaligned_x(ig3):
    # x at a 4-byte offset: AUTO takes the FMA kernel, TC refuses (the tensor-map copy
    # needs a 16-byte aligned base).
    N, Cin, D, H, W, Cout, pad = 1, 8, 6, 8, 16, 32, 1
    wl = si.conv3d_workload("t", N, Cin, D, H, W, Cout, seed=3390, epilogue="tanh_mish", pad=pad)
    t = wl.generate_all()
    flat = torch.zeros(t["x"].size + 1, dtype=torch.float32, device="cuda")
    flat[1:] = to_dev(t["x"]).reshape(-1)
    x = flat[1:].view(t["x"].shape)
    assert x.data_ptr() % 16 != 0
    ref = oracle.tanh_mish(oracle.conv3d_ex(t["x"], t["w"], t["b"], pad, 2))
    got = ig3.conv3d_fused(x, to_dev(t["w"]), to_dev(t["b"]), epilogue="tanh_mish", pad=pad, stride=2)
    assert_close(got.cpu().numpy(), ref, "misaligned x, auto")
    with pytest.raises(RuntimeError):
        ig3.conv3d_fused(x, to_dev(t["w"]), to_dev(t["b"]), epilogue="tanh_mish", path="tc", pad=pad, stride=2)


def test_conv3d_stride2_full_size_sampled(ig3):
    wl = si.conv3d_stride2_tanh_mish()
    t = wl.generate_all()
    x = to_dev(t["x"]); w = to_dev(t["w"]); b = to_dev(t["b"])
    out = ig3.conv3d_fused(x, w, b, epilogue="tanh_mish", pad=wl.pad, stride=wl.stride)   # the benchmark's call
    assert ig3.ig3_last_device_status() == 0
    assert tuple(out.shape) == (16, 64, 16, 32, 32)
    idx = sample_indices(tuple(out.shape), 6000, seed=71)
    got = out[tuple(torch.from_numpy(idx.T).to(out.device))].cpu().numpy()
    ref = oracle.tanh_mish(oracle.conv3d_ex_at(t["x"], t["w"], t["b"], wl.pad, wl.stride, idx))
    assert_close(got, ref, "conv3d stride 2 full size sampled")
    del x, w, b, out
    torch.cuda.empty_cache()
