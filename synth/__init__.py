"""Seeded synthetic inputs for the INT8 NCxHWx<32> convolution workloads and
the fp32 direct-convolution workload.

This module is shared by the CPU oracle's tests and by the GPU path's tests and
benchmark. It holds only random-number generation and the workload table; it
contains none of the convolution's arithmetic (no output-size formula, no
layout transform, no accumulation), so neither side can borrow method code
from the other through it.

Generator: xoshiro256** (Blackman & Vigna, "Scrambled linear pseudorandom
number generators", 2018), each lane seeded from one SplitMix64 stream
(Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
2014).  To generate tens of millions of values quickly in numpy the stream is
split into ``LANES`` independent xoshiro256** lanes: element ``j`` of a draw
of length ``n`` is output number ``j // LANES`` of lane ``j % LANES``.  Lane
``i`` takes words ``4i .. 4i+3`` of the SplitMix64 sequence that starts at the
seed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

LANES = 1 << 16
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _u64(v: int) -> np.uint64:
    return np.uint64(v & 0xFFFFFFFFFFFFFFFF)


def splitmix64(seed: int, count: int) -> np.ndarray:
    """Words 1..count of the SplitMix64 sequence started at ``seed``."""
    k = np.arange(1, count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _u64(seed) + k * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _rotl(x: np.ndarray, k: int) -> np.ndarray:
    return (x << np.uint64(k)) | (x >> np.uint64(64 - k))


class Xoshiro256ss:
    """``LANES`` parallel xoshiro256** generators seeded from one SplitMix64 stream."""

    def __init__(self, seed: int, lanes: int = LANES):
        words = splitmix64(seed, 4 * lanes).reshape(lanes, 4)
        self.s = [words[:, i].copy() for i in range(4)]
        self.lanes = lanes

    def _step(self) -> np.ndarray:
        s0, s1, s2, s3 = self.s
        with np.errstate(over="ignore"):
            out = _rotl(s1 * np.uint64(5), 7) * np.uint64(9)
        t = s1 << np.uint64(17)
        s2 ^= s0
        s3 ^= s1
        s1 ^= s2
        s0 ^= s3
        s2 ^= t
        self.s = [s0, s1, s2, _rotl(s3, 45)]
        return out

    def next_u64(self, n: int) -> np.ndarray:
        """``n`` 64-bit outputs; element j comes from lane j % lanes."""
        steps = -(-n // self.lanes)
        out = np.empty(steps * self.lanes, dtype=np.uint64)
        for d in range(steps):
            out[d * self.lanes:(d + 1) * self.lanes] = self._step()
        return out[:n]


def uniform_int8(seed: int, count: int, lo: int, hi: int) -> np.ndarray:
    """``count`` int8 values uniform on [lo, hi]: lo + ((u >> 32) * span) >> 32."""
    if not (-128 <= lo <= hi <= 127):
        raise ValueError("range must lie inside int8")
    span = np.uint64(hi - lo + 1)
    u = Xoshiro256ss(seed).next_u64(count)
    v = ((u >> np.uint64(32)) * span) >> np.uint64(32)
    return (v.astype(np.int64) + lo).astype(np.int8)


def normal_int8(seed: int, count: int, sigma: float) -> np.ndarray:
    """``count`` int8 values: round-half-even(sigma * z) clamped to [-128, 127].

    z is a standard normal from the Box-Muller transform of draw pairs
    (u[2i], u[2i+1]): u1 = ((u[2i] >> 11) + 1) / 2^53 in (0, 1],
    u2 = (u[2i+1] >> 11) / 2^53 in [0, 1), z = sqrt(-2 ln u1) cos(2 pi u2).
    """
    u = Xoshiro256ss(seed).next_u64(2 * count)
    scale = 1.0 / float(1 << 53)
    u1 = ((u[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * scale
    u2 = (u[1::2] >> np.uint64(11)).astype(np.float64) * scale
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return np.clip(np.rint(sigma * z), -128, 127).astype(np.int8)


def uniform_f32(seed: int, count: int, lo: float, hi: float) -> np.ndarray:
    """``count`` float32 values uniform on [lo, hi): lo + (hi - lo) * (u >> 40) / 2^24,
    computed in double and rounded once to float32."""
    u = Xoshiro256ss(seed).next_u64(count)
    t = (u >> np.uint64(40)).astype(np.float64) * (1.0 / float(1 << 24))
    return (lo + (hi - lo) * t).astype(np.float32)


@dataclass(frozen=True)
class F32Workload:
    """The fp32 direct convolution of the kernel-benchmark trace (nn.Conv2d
    on NCHW fp32): inputs uniform on [0, 1), weights and bias uniform on
    [-b, b) with b = 1/sqrt(C*R*S) (nn.Conv2d's default initialisation bound)."""
    name: str
    N: int
    C: int
    H: int
    W: int
    K: int
    R: int
    S: int
    pad: tuple
    stride: tuple
    dil: tuple
    seed: int

    def shape_tuple(self):
        return (self.N, self.C, self.H, self.W, self.K, self.R, self.S, self.pad[0], self.pad[1],
                self.stride[0], self.stride[1], self.dil[0], self.dil[1])

    def bound(self) -> float:
        return 1.0 / math.sqrt(self.C * self.R * self.S)

    def inputs_nchw(self) -> np.ndarray:
        return uniform_f32(self.seed, self.N * self.C * self.H * self.W, 0.0, 1.0).reshape(
            self.N, self.C, self.H, self.W)

    def weights_kcrs(self) -> np.ndarray:
        b = self.bound()
        return uniform_f32(self.seed + 1, self.K * self.C * self.R * self.S, -b, b).reshape(
            self.K, self.C, self.R, self.S)

    def bias(self) -> np.ndarray:
        b = self.bound()
        return uniform_f32(self.seed + 2, self.K, -b, b)


# page 4's problem: batch 8, 32 -> 64 channels, 512 x 512, 5 x 9 kernel, pad (2, 4), dilation (2, 3)
F32_WORKLOAD = F32Workload("f32_n8c32h512k64r5x9d2x3", 8, 32, 512, 512, 64, 5, 9, (2, 4), (1, 1), (2, 3), 20260200)


@dataclass(frozen=True)
class Workload:
    """One convolution workload: shapes, value distribution, alpha and seeds.

    Tensor values are drawn in logical NCHW order (activations) and KCRS order
    (filters): element (n, c, h, w) is draw number ((n*C + c)*H + h)*W + w.
    """

    name: str
    N: int
    C: int
    H: int
    W: int
    K: int
    R: int
    S: int
    pad_h: int
    pad_w: int
    stride_h: int
    stride_w: int
    dil_h: int
    dil_w: int
    alpha: float
    dist: str  # "uniform:lo:hi" or "normal:sigma"
    x_seed: int
    f_seed: int

    def shape_tuple(self):
        return (self.N, self.C, self.H, self.W, self.K, self.R, self.S,
                self.pad_h, self.pad_w, self.stride_h, self.stride_w,
                self.dil_h, self.dil_w)

    def _draw(self, seed: int, count: int) -> np.ndarray:
        kind, *args = self.dist.split(":")
        if kind == "uniform":
            return uniform_int8(seed, count, int(args[0]), int(args[1]))
        if kind == "normal":
            return normal_int8(seed, count, float(args[0]))
        raise ValueError(self.dist)

    def activations_nchw(self) -> np.ndarray:
        n = self.N * self.C * self.H * self.W
        return self._draw(self.x_seed, n).reshape(self.N, self.C, self.H, self.W)

    def filters_kcrs(self) -> np.ndarray:
        n = self.K * self.C * self.R * self.S
        return self._draw(self.f_seed, n).reshape(self.K, self.C, self.R, self.S)


def _wl(i, name, N, C, H, W, K, R, S, pad, stride, dil, alpha, dist):
    return Workload(name, N, C, H, W, K, R, S, pad[0], pad[1], stride[0], stride[1],
                    dil[0], dil[1], alpha, dist, 20260000 + i, 20260100 + i)


# The five workloads: a 16x16 single-image 3x3 layer, two ResNet-style 3x3
# layers (one strided), the 5x9 dilated layer of the kernel-benchmark problem
# on page 4, and a wide 28x28 3x3 layer with normally distributed values.
WORKLOADS = [
    _wl(1, "n1c32h16k32r3s1", 1, 32, 16, 16, 32, 3, 3, (1, 1), (1, 1), (1, 1), 2.0 ** -9, "uniform:-128:127"),
    _wl(2, "n8c256h56k256r3s1", 8, 256, 56, 56, 256, 3, 3, (1, 1), (1, 1), (1, 1), 2.0 ** -12, "uniform:-128:127"),
    _wl(3, "n32c128h112k256r3s2", 32, 128, 112, 112, 256, 3, 3, (1, 1), (2, 2), (1, 1), 2.0 ** -10, "uniform:-64:63"),
    _wl(4, "n8c32h512k64r5x9d2x3", 8, 32, 512, 512, 64, 5, 9, (2, 4), (1, 1), (2, 3), 2.0 ** -11, "uniform:-128:127"),
    _wl(5, "n64c512h28k512r3s1", 64, 512, 28, 28, 512, 3, 3, (1, 1), (1, 1), (1, 1), 2.0 ** -13, "normal:32"),
]
WORKLOADS_BY_NAME = {w.name: w for w in WORKLOADS}
