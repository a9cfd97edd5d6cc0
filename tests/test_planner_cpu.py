"""The tensor-core planners and the addresses their kernels derive, checked on the host.

tests/planner_check.cu includes the conv3d planner (csrc/conv3d_tc.cu) and, for every
work unit of every CTA, recomputes the indices the kernel uses (TMEM columns, slots, B
blocks, A rows, shared-memory offsets, input copies) against the plan's buffers;
tests/tc16_plan_check.cu does the same for the 16-output-channel kernel with A in tensor
memory (slot ring and its wrapped runs, A stages, B blocks, raw input copies, partials);
tests/strided_tc_plan_check.cu does it for the stride-2 kernel (every gathered box
element against the input coordinate of the definition, copies, columns, coverage);
tests/dwsep_plan_check.cu does the same for the depthwise-separable planner (strips,
shared-memory layout, TMEM ranges, tensor-map box and strides, row-copy coordinates).
They need nvcc (host compilation only) but no GPU.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.parametrize("checker", ["planner_check.cu", "tc16_plan_check.cu", "strided_tc_plan_check.cu",
                                     "dwsep_plan_check.cu"])
def test_planner_index_bounds(checker):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, checker[:-3])
        cmd = [nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
               "-I" + os.path.join(ROOT, "include"), "-o", exe, os.path.join(HERE, checker),
               "-Xlinker", "--unresolved-symbols=ignore-all"]
        b = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
        assert b.returncode == 0, b.stderr[-2000:]
        r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:]
    assert "fails: 0" in r.stdout
