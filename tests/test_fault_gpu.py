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
