"""Failure detection on the GPU without a GPU fault: a bounded wait runs out on a
barrier nothing completes, the kernel returns, the host reads the status, and
the context stays usable."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ig3():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_x3x3_gb300 as m
    return m


def test_bounded_wait_times_out_and_context_survives(ig3):
    assert ig3.ig3_last_device_status() == 0
    ig3.ig3_selftest_bounded_wait(2_000_000)  # 2 ms limit
    assert ig3.ig3_last_device_status() == -4  # IG3_ERR_TIMEOUT
    assert ig3.ig3_last_device_status() == 0   # reading clears it
    # The context still works: a normal call succeeds afterwards.
    x = torch.randn(1, 4, 5, 6, 7, device="cuda")
    w = torch.randn(8, 4, 3, 3, 3, device="cuda")
    y = ig3.conv3d_fused(x, w, None, epilogue="none", path="fma")
    torch.cuda.synchronize()
    assert ig3.ig3_last_device_status() == 0
    assert bool(torch.isfinite(y).all())


def test_launch_counter_moves(ig3):
    before = ig3.ig3_kernel_launches()
    x = torch.randn(1, 4, 5, 6, 7, device="cuda")
    w = torch.randn(8, 4, 3, 3, 3, device="cuda")
    ig3.conv3d_fused(x, w, None, epilogue="none", path="fma")
    torch.cuda.synchronize()
    assert ig3.ig3_kernel_launches() == before + 1


def test_tensor_core_kernels_abort_and_recover(ig3):
    # A 1 ns wait limit makes the first wait that has to spin give up (waits that
    # sleep in the barrier look at the limit every ~20 us, so the shapes are large
    # enough for some wait to last that long): the kernels' abort path runs (every role stops, in-flight copies and MMAs drain with their
    # own 1 s floor, tensor memory is freed), the status reports the timeout, and a
    # normal call afterwards gives the oracle's result.
    import oracle
    import seeded_inputs as si
    from parity import assert_close, to_dev
    conv_cases = [
        ("conv Cout 16 (A in tensor memory)", (4, 16, 12, 32, 64, 16), "tanh_mish"),
        ("pool-reduce Cout 16", (32, 8, 10, 34, 64, 16), "pool_reduce"),
        ("conv Cout 64", (2, 32, 8, 20, 64, 64), "tanh_mish"),
    ]
    try:
        for name, (N, Cin, D, H, W, Cout), epi in conv_cases:
            wl = si.conv3d_workload("abort", N, Cin, D, H, W, Cout, seed=4300 + Cout + Cin, epilogue=epi,
                                    bias2=(epi == "pool_reduce"))
            t = wl.generate_all()
            dev = {k: to_dev(v) for k, v in t.items()}
            params = {"divisor": 2.0, "pool": 2, "bias2": dev["bias2"]} if epi == "pool_reduce" else None
            ig3.ig3_set_wait_timeout_ns(1)
            ig3.conv3d_fused(dev["x"], dev["w"], dev["b"], epilogue=epi, params=params, path="tc")
            assert ig3.ig3_last_device_status() == -4, name  # IG3_ERR_TIMEOUT
            ig3.ig3_set_wait_timeout_ns(0)                   # back to the default limit
            got = ig3.conv3d_fused(dev["x"], dev["w"], dev["b"], epilogue=epi, params=params, path="tc")
            assert ig3.ig3_last_device_status() == 0, name
            if epi == "pool_reduce":
                ref = oracle.conv3d_pool_reduce(t["x"], t["w"], t["b"], 2.0, 2, t["bias2"])
            else:
                ref = oracle.conv3d_tanh_mish(t["x"], t["w"], t["b"])
            assert_close(got.cpu().numpy(), ref, f"{name} after an aborted call")
        wl = si.conv3d_workload("abort_s2", 2, 32, 16, 64, 64, 64, seed=4350, epilogue="tanh_mish", pad=1)
        t = wl.generate_all()
        dev = {k: to_dev(v) for k, v in t.items()}
        ig3.ig3_set_wait_timeout_ns(1)
        ig3.conv3d_fused(dev["x"], dev["w"], dev["b"], epilogue="tanh_mish", path="tc", pad=1, stride=2)
        assert ig3.ig3_last_device_status() == -4, "stride 2"
        ig3.ig3_set_wait_timeout_ns(0)
        got = ig3.conv3d_fused(dev["x"], dev["w"], dev["b"], epilogue="tanh_mish", path="tc", pad=1, stride=2)
        assert ig3.ig3_last_device_status() == 0
        assert_close(got.cpu().numpy(), oracle.tanh_mish(oracle.conv3d_ex(t["x"], t["w"], t["b"], 1, 2)),
                     "stride 2 after an aborted call")
        wl = si.dwsep_workload("abort_dwsep", 2, 32, 64, 128, 64, seed=4400)
        t = wl.generate_all()
        dev = {k: to_dev(v) for k, v in t.items()}
        ig3.ig3_set_wait_timeout_ns(1)
        ig3.dwsep_conv2d(dev["x"], dev["w_dw"], dev["w_pw"], None, path="tc")
        assert ig3.ig3_last_device_status() == -4, "dwsep"
        ig3.ig3_set_wait_timeout_ns(0)
        got = ig3.dwsep_conv2d(dev["x"], dev["w_dw"], dev["w_pw"], None, path="tc")
        assert ig3.ig3_last_device_status() == 0
        assert_close(got.cpu().numpy(), oracle.dwsep(t["x"], t["w_dw"], t["w_pw"], None), "dwsep after an aborted call")
        wl = si.dwsep_workload("abort_dwsep5", 2, 32, 64, 128, 64, seed=4410, K=5)
        t = wl.generate_all()
        dev = {k: to_dev(v) for k, v in t.items()}
        ig3.ig3_set_wait_timeout_ns(1)
        ig3.dwsep_conv2d(dev["x"], dev["w_dw"], dev["w_pw"], None, path="tc")
        assert ig3.ig3_last_device_status() == -4, "dwsep K=5"
        ig3.ig3_set_wait_timeout_ns(0)
        got = ig3.dwsep_conv2d(dev["x"], dev["w_dw"], dev["w_pw"], None, path="tc")
        assert ig3.ig3_last_device_status() == 0
        assert_close(got.cpu().numpy(), oracle.dwsep_k(t["x"], t["w_dw"], t["w_pw"], None),
                     "dwsep K=5 after an aborted call")
    finally:
        ig3.ig3_set_wait_timeout_ns(0)
        ig3.ig3_last_device_status()
