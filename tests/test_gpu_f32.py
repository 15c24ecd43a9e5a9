"""GPU parity of the fp32 direct convolution (the kernel-benchmark trace's
nn.Conv2d) against the double-precision oracle.

Two bars: the trace's own checker tolerance, |y - ref| <= 1e-4 + 1e-4 * |ref|
(read from the page-4 golden fixture, with its citation), and the rigorous
fp32 summation bound, |y - ref| <=
gamma_{C*R*S+1} * (|bias| + sum |x * w|) with unit roundoff 2^-24, which holds
for any order of fp32 additions and fused multiply-adds and is far tighter on
small sums.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 3, 17, 23, 5, 3, 3, 1, 1, 1, 1, 1, 1),      # C, K not multiples of anything; ragged tiles
    (2, 32, 40, 44, 64, 5, 9, 2, 4, 1, 1, 2, 3),    # the trace's layer geometry, small image
    (1, 7, 33, 35, 70, 3, 5, 0, 2, 2, 1, 1, 2),     # K past one 64-channel tile, stride 2 rows
    (2, 5, 19, 41, 9, 2, 4, 1, 0, 1, 3, 3, 1),      # column stride 3, row dilation 3
    (1, 1, 8, 8, 1, 1, 1, 0, 0, 1, 1, 1, 1),        # 1x1 filter, one channel
    (1, 4, 9, 70, 3, 1, 7, 0, 3, 2, 2, 1, 4),       # several column tiles, wide dilation
]


def _data(shape, seed):
    N, C, H, W, K, R, S = shape[:7]
    b = 1.0 / np.sqrt(C * R * S)
    x = synth.uniform_f32(seed, N * C * H * W, 0.0, 1.0).reshape(N, C, H, W)
    w = synth.uniform_f32(seed + 1, K * C * R * S, -b, b).reshape(K, C, R, S)
    bias = synth.uniform_f32(seed + 2, K, -b, b)
    return x, w, bias


def _page4_tolerance():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "page4_dilated_conv.json")) as fh:
        t = json.load(fh)["checker_tolerance"]
    return t["atol"], t["rtol"]


def _check(y, ref, mag, terms):
    orc = oracle.Oracle()
    diff = np.abs(y.astype(np.float64) - ref)
    assert np.all(diff <= orc.f32_error_bound(mag, terms)), float(np.max(diff))
    atol, rtol = _page4_tolerance()
    assert np.all(diff <= atol + rtol * np.abs(ref))


@pytest.mark.parametrize("with_bias", [True, False], ids=["bias", "no-bias"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_f32_direct_matches_oracle(shape, with_bias):
    import torch
    import int8_implicit_gemm_gb300 as ext
    x, w, bias = _data(shape, 500 + sum(shape))
    b = bias if with_bias else None
    ref, mag = oracle.Oracle().conv_f64(x, w, shape, bias=b)
    y = ext.conv2d_fprop_f32(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), shape,
                             bias=None if b is None else torch.from_numpy(b).cuda())
    torch.cuda.synchronize()
    assert tuple(y.shape) == ref.shape
    _check(y.cpu().numpy(), ref, mag, shape[1] * shape[5] * shape[6])


def test_f32_direct_full_size_page4_layer():
    """The trace's layer at full size (8 x 32 x 512 x 512 -> 8 x 64 x 508 x 496),
    bias included: sampled outputs (random ones plus every border and corner
    region) against the oracle point by point."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    wl = synth.F32_WORKLOAD
    shape = wl.shape_tuple()
    x, w, bias = wl.inputs_nchw(), wl.weights_kcrs(), wl.bias()
    y = ext.conv2d_fprop_f32(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), shape,
                             bias=torch.from_numpy(bias).cuda())
    torch.cuda.synchronize()
    N, K, P, Q = y.shape
    assert (P, Q) == (508, 496)
    rng = np.random.default_rng(9)
    pts = [(rng.integers(N), rng.integers(K), rng.integers(P), rng.integers(Q)) for _ in range(1500)]
    for p in (0, 1, 2, P // 2, P - 3, P - 2, P - 1):
        for q in (0, 1, 3, 4, 5, Q // 2, Q - 6, Q - 5, Q - 2, Q - 1):
            pts.append((rng.integers(N), rng.integers(K), p, q))
    pts = np.array(pts, dtype=np.int64)
    ref, mag = oracle.Oracle().conv_f64_points(x, w, shape, pts, bias=bias)
    yv = y.cpu().numpy()[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
    _check(yv, ref, mag, wl.C * wl.R * wl.S)


def test_f32_direct_argument_errors():
    import ctypes
    import torch
    import int8_implicit_gemm_gb300 as ext
    shape = (1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 1, 1)
    x = torch.zeros(1 * 3 * 64 + 1, device="cuda")
    w = torch.zeros(4 * 3 * 9, device="cuda")
    y = torch.zeros(4 * 64 + 1, device="cuda")
    sh = ctypes.byref(ext.ConvShape.of(shape))
    f = ext.lib.i8c_conv2d_fprop_f32
    assert f(x.data_ptr() + 2, w.data_ptr(), None, y.data_ptr(), sh, None) == ext.I8C_ERR_MISALIGNED
    assert f(None, w.data_ptr(), None, y.data_ptr(), sh, None) == ext.I8C_ERR_INVALID_ARG
    bad = ctypes.byref(ext.ConvShape.of((1, 3, 2, 2, 4, 5, 5, 0, 0, 1, 1, 1, 1)))
    assert f(x.data_ptr(), w.data_ptr(), None, y.data_ptr(), bad, None) == ext.I8C_ERR_UNSUPPORTED
    # a valid call on the same buffers still works afterwards
    assert f(x.data_ptr(), w.data_ptr(), None, y.data_ptr(), sh, None) == 0
    torch.cuda.synchronize()
    assert float(y[:4 * 64].abs().max()) == 0.0
