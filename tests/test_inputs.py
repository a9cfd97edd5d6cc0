"""The seeded input generator: SplitMix64 against its published outputs, and the
distributions, counters and workload recipes built on it."""
import math

import numpy as np
import pytest

import seeded_inputs as si


def test_splitmix64_published_outputs():
    # The first three outputs of SplitMix64 from state 0 (Vigna's reference splitmix64.c).
    assert [si.splitmix64_scalar(0, k) for k in range(3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_vector_matches_scalar():
    for seed in (0, 3, 2**63 + 5):
        v = si.splitmix64(seed, 1000, 17)
        assert [int(z) for z in v] == [si.splitmix64_scalar(seed, 1000 + i) for i in range(17)]


def test_counter_form_allows_random_access():
    full = si.draw(7, 0, (1000,), ("normal",))
    part = si.draw(7, 300, (200,), ("normal",))
    assert np.array_equal(full[300:500], part)


def test_uniform_bounds_and_moments():
    u = si.draw(11, 0, (1 << 20,), ("uniform", -0.25, 0.25))
    assert u.dtype == np.float32 and u.min() >= -0.25 and u.max() <= 0.25
    assert abs(u.mean()) < 2e-3 and abs(u.std() - 0.5 / math.sqrt(12)) < 1e-3


def test_normal_moments():
    n = si.draw(12, 0, (1 << 20,), ("normal",)).astype(np.float64)
    assert abs(n.mean()) < 5e-3 and abs(n.std() - 1.0) < 5e-3
    assert abs((n ** 3).mean()) < 2e-2 and abs((n ** 4).mean() - 3.0) < 5e-2


def test_workload_draw_order_and_shapes():
    wl = si.conv3d_pool_reduce()
    assert [t.name for t in wl.tensors] == ["x", "w", "b", "bias2"]
    assert wl.spec("x").shape == (128, 8, 16, 64, 64)
    assert wl.offset("w") == wl.spec("x").numel
    assert wl.offset("bias2") == wl.spec("x").numel + wl.spec("w").numel + 16
    assert wl.dims == dict(N=128, Cin=8, D=16, H=64, W=64, Cout=16)
    a = 1 / math.sqrt(216)
    assert wl.spec("w").dist == ("uniform", -a, a)


def test_tiny_workload():
    wl = si.tiny_conv3d()
    t = wl.generate_all()
    assert wl.seed == 0
    assert t["x"].shape == (2, 4, 8, 8, 8) and t["x"].min() >= -1 and t["x"].max() <= 1
    a = 1 / math.sqrt(108)
    assert np.abs(t["w"]).max() <= a and np.abs(t["b"]).max() <= a


@pytest.mark.parametrize("wl", si.all_workloads(), ids=lambda w: w.name)
def test_every_workload_is_well_formed(wl):
    names = [t.name for t in wl.tensors]
    assert names[0] == "x"
    if wl.op == "conv3d":
        d = wl.dims
        assert wl.spec("w").shape == (d["Cout"], d["Cin"], 3, 3, 3)
    else:
        d = wl.dims
        assert wl.spec("w_dw").shape == (d["C"], 1, d["K"], d["K"]) and d["K"] in (1, 3, 5, 7)
        assert wl.spec("w_pw").shape == (d["Cout"], d["C"], 1, 1)
