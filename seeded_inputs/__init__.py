"""Seeded synthetic inputs for the fused 3x3(x3) convolution workloads.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It holds no arithmetic of the convolution method itself: it only
draws random numbers and knows the workload shapes and distributions.

Generator
---------
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), used in its counter form: the k-th 64-bit output
(k = 0, 1, 2, ...) of a stream with seed ``s`` is ``mix(s + (k + 1) * GAMMA)``
with ``GAMMA = 0x9E3779B97F4A7C15`` and ``mix`` the published finaliser
(xor-shift 30, multiply 0xBF58476D1CE4E5B9, xor-shift 27, multiply
0x94D049BB133111EB, xor-shift 31).  Because every draw is a pure function of its
counter, any element of any tensor can be regenerated on its own.

Draw order: one stream per workload; tensors are drawn one after the other in
the listed order, tensor ``t`` taking the counters ``[offset_t, offset_t +
numel_t)`` where ``offset_t`` is the total size of the tensors before it.

Distributions (each value computed in float64, then rounded to float32):

* ``U[a, b)``: ``u = (z >> 40) * 2**-24``; value ``a + (b - a) * u``.
* ``N(0, 1)``: Box-Muller on one 64-bit draw, ``u1 = ((z >> 32) + 0.5) / 2**32``,
  ``u2 = (z & 0xFFFFFFFF) / 2**32``, value ``sqrt(-2 ln u1) * cos(2 pi u2)``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1

_CHUNK = 1 << 22  # elements generated per numpy pass (bounds temporary memory)


def splitmix64_scalar(seed: int, k: int) -> int:
    """k-th output of the SplitMix64 stream with the given seed (pure Python)."""
    z = (seed + (k + 1) * GAMMA) & _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the stream, as a uint64 array."""
    k = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    z = k * np.uint64(GAMMA)
    z += np.uint64(seed & _MASK64)
    z ^= z >> np.uint64(30)
    z *= np.uint64(_M1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(_M2)
    z ^= z >> np.uint64(31)
    return z


def _uniform_from(z: np.ndarray, lo: float, hi: float) -> np.ndarray:
    u = (z >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
    return (lo + (hi - lo) * u).astype(np.float32)


def _normal_from(z: np.ndarray) -> np.ndarray:
    u1 = ((z >> np.uint64(32)).astype(np.float64) + 0.5) * (2.0 ** -32)
    u2 = (z & np.uint64(0xFFFFFFFF)).astype(np.float64) * (2.0 ** -32)
    return (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)).astype(np.float32)


def draw(seed: int, offset: int, shape, dist: tuple, out: np.ndarray | None = None) -> np.ndarray:
    """Draw a float32 tensor of ``shape`` from counters ``offset ..``.

    ``dist`` is ``("uniform", lo, hi)`` or ``("normal",)``.  ``out`` may be a
    preallocated (e.g. pinned) float32 array of the right size to fill in place.
    """
    n = int(np.prod(shape, dtype=np.int64))
    if out is None:
        out = np.empty(n, dtype=np.float32)
    flat = out.reshape(-1)
    if flat.size != n:
        raise ValueError("out has the wrong size")
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        z = splitmix64(seed, offset + s, c)
        if dist[0] == "uniform":
            flat[s:s + c] = _uniform_from(z, dist[1], dist[2])
        elif dist[0] == "normal":
            flat[s:s + c] = _normal_from(z)
        else:
            raise ValueError(f"unknown distribution {dist!r}")
    return out.reshape(shape)


@dataclass
class TensorSpec:
    name: str
    shape: tuple
    dist: tuple

    @property
    def numel(self) -> int:
        return int(np.prod(self.shape, dtype=np.int64))


@dataclass
class Workload:
    """One synthetic workload: op kind, tensors in draw order, seed, op parameters."""
    name: str
    op: str                      # "conv3d" or "dwsep"
    seed: int
    tensors: list = field(default_factory=list)
    epilogue: str = "none"       # conv3d only: "none" | "tanh_mish" | "pool_reduce"
    divisor: float = 2.0         # pool_reduce only
    pool: int = 2                # pool_reduce only
    pad: int = 0                 # conv3d only: zero padding on every side
    stride: int = 1              # conv3d only

    def spec(self, name: str) -> TensorSpec:
        for t in self.tensors:
            if t.name == name:
                return t
        raise KeyError(name)

    def offset(self, name: str) -> int:
        off = 0
        for t in self.tensors:
            if t.name == name:
                return off
            off += t.numel
        raise KeyError(name)

    def generate(self, name: str, out: np.ndarray | None = None) -> np.ndarray:
        t = self.spec(name)
        return draw(self.seed, self.offset(name), t.shape, t.dist, out=out)

    def generate_all(self) -> dict:
        return {t.name: self.generate(t.name) for t in self.tensors}

    @property
    def dims(self) -> dict:
        if self.op == "conv3d":
            n, cin, d, h, w = self.spec("x").shape
            cout = self.spec("w").shape[0]
            return dict(N=n, Cin=cin, D=d, H=h, W=w, Cout=cout)
        n, c, h, w = self.spec("x").shape
        cout = self.spec("w_pw").shape[0]
        return dict(N=n, C=c, H=h, W=w, Cout=cout, K=self.spec("w_dw").shape[-1])


def _u(a: float) -> tuple:
    return ("uniform", -a, a)


NORMAL = ("normal",)


def conv3d_workload(name, N, Cin, D, H, W, Cout, seed, epilogue="tanh_mish",
                    x_dist=NORMAL, with_bias=True, bias2=False, wb_bound=None, pad=0, stride=1) -> Workload:
    """Conv3d workload: x ~ x_dist, w and b ~ U(+-1/sqrt(27*Cin)) unless wb_bound given."""
    a = wb_bound if wb_bound is not None else 1.0 / math.sqrt(27.0 * Cin)
    ts = [TensorSpec("x", (N, Cin, D, H, W), x_dist),
          TensorSpec("w", (Cout, Cin, 3, 3, 3), _u(a))]
    if with_bias:
        ts.append(TensorSpec("b", (Cout,), _u(a)))
    if bias2:
        ts.append(TensorSpec("bias2", (Cout,), NORMAL))
    return Workload(name=name, op="conv3d", seed=seed, tensors=ts, epilogue=epilogue, pad=pad, stride=stride)


def dwsep_workload(name, N, C, H, W, Cout, seed, x_dist=NORMAL, with_bias=False, K=3) -> Workload:
    """Depthwise KxK ("same" padding) then pointwise 1x1: w_dw ~ U(+-1/K), w_pw ~ U(+-1/sqrt(C))."""
    ts = [TensorSpec("x", (N, C, H, W), x_dist),
          TensorSpec("w_dw", (C, 1, K, K), _u(1.0 / K)),
          TensorSpec("w_pw", (Cout, C, 1, 1), _u(1.0 / math.sqrt(C)))]
    if with_bias:
        ts.append(TensorSpec("b", (Cout,), _u(1.0 / math.sqrt(C))))
    return Workload(name=name, op="dwsep", seed=seed, tensors=ts)


# The five benchmark workloads.  Seeds: the tiny case uses seed 0; the others use
# their 1-based config number; the channel sweep uses 500 + C.
def tiny_conv3d() -> Workload:
    """x[2,4,8,8,8] ~ U(-1,1); w[8,4,3,3,3], b[8] ~ U(+-1/sqrt(108)); tanh(mish)."""
    return conv3d_workload("tiny_conv3d_tanh_mish", 2, 4, 8, 8, 8, 8, seed=0,
                           epilogue="tanh_mish", x_dist=("uniform", -1.0, 1.0))


def conv3d_tanh_mish() -> Workload:
    """x[16,32,32,64,64] ~ N(0,1); w[64,32,3,3,3], b[64] ~ U(+-1/sqrt(864))."""
    return conv3d_workload("conv3d_tanh_mish_16x32x32x64x64_c64", 16, 32, 32, 64, 64, 64,
                           seed=2, epilogue="tanh_mish")


def conv3d_pool_reduce() -> Workload:
    """x[128,8,16,64,64] ~ N(0,1); w[16,8,3,3,3], b[16] ~ U(+-1/sqrt(216)); bias2[16] ~ N(0,1)."""
    return conv3d_workload("conv3d_pool_reduce_128x8x16x64x64_c16", 128, 8, 16, 64, 64, 16,
                           seed=3, epilogue="pool_reduce", bias2=True)


def dwsep_conv2d() -> Workload:
    """x[16,64,512,512] ~ N(0,1); w_dw[64,1,3,3] ~ U(+-1/3); w_pw[128,64,1,1] ~ U(+-1/8)."""
    return dwsep_workload("dwsep_16x64x512x512_c128", 16, 64, 512, 512, 128, seed=4)


def conv3d_sweep(C: int) -> Workload:
    """x[8,C,32,64,64] ~ N(0,1); w, b ~ U(+-1/sqrt(27*C)); Cout = C; tanh(mish)."""
    return conv3d_workload(f"conv3d_tanh_mish_sweep_8x{C}x32x64x64_c{C}", 8, C, 32, 64, 64, C,
                           seed=500 + C, epilogue="tanh_mish")


def conv3d_same_tanh_mish() -> Workload:
    """The conv3d + tanh(mish) workload with zero padding 1 (output [16,64,32,64,64]); seed 6."""
    return conv3d_workload("conv3d_same_tanh_mish_16x32x32x64x64_c64", 16, 32, 32, 64, 64, 64,
                           seed=6, epilogue="tanh_mish", pad=1)


def conv3d_stride2_tanh_mish() -> Workload:
    """The conv3d + tanh(mish) input with padding 1 and stride 2 (output [16,64,16,32,32]); seed 7."""
    return conv3d_workload("conv3d_s2_tanh_mish_16x32x32x64x64_c64", 16, 32, 32, 64, 64, 64,
                           seed=7, epilogue="tanh_mish", pad=1, stride=2)


def dwsep_k5() -> Workload:
    """The dwsep input with a 5x5 depthwise stage (padding 2): x[16,64,512,512] -> 128; seed 8."""
    return dwsep_workload("dwsep_k5_16x64x512x512_c128", 16, 64, 512, 512, 128, seed=8, K=5)


def all_workloads() -> list:
    return [tiny_conv3d(), conv3d_tanh_mish(), conv3d_pool_reduce(), dwsep_conv2d(),
            conv3d_sweep(16), conv3d_sweep(64), conv3d_sweep(128), conv3d_same_tanh_mish(),
            conv3d_stride2_tanh_mish(), dwsep_k5()]
