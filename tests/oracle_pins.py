"""Pins for the CPU oracle: checks against values the pages print, closed forms,
brute force and an independent library routine -- never against the oracle
itself.  Each ``pin_*`` takes an ``oracle.Oracle`` handle and raises
``AssertionError`` on a mismatch, so the same pins run against the real
oracle and against variants with planted mistakes (tests/test_oracle_mutants.py).
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _page4():
    with open(os.path.join(GOLDEN, "page4_dilated_conv.json")) as fh:
        return json.load(fh)


def _shape_of(d):
    return (d["N"], d["C"], d["H"], d["W"], d["K"], d["R"], d["S"],
            d["pad_h"], d["pad_w"], d["stride_h"], d["stride_w"], d["dil_h"], d["dil_w"])


# --- output extent -----------------------------------------------------------

def pin_output_size_page4(orc):
    """Page 4 prints the 508x496 output of its 5x9 dilated layer."""
    g = _page4()
    assert orc.out_size(_shape_of(g["shape"])) == (g["output_size"]["P"], g["output_size"]["Q"])


def pin_output_size_bruteforce(orc):
    """Extent = number of window positions p >= 0 whose dilated window,
    stepped by the stride, ends inside the zero-padded input (counted)."""
    for size in (1, 2, 5, 7, 16, 28):
        for pad in (0, 1, 2, 4):
            for dil in (1, 2, 3):
                for k in (1, 3, 5):
                    for stride in (1, 2, 3):
                        padded = size + 2 * pad
                        count = 0
                        while count * stride + dil * (k - 1) < padded:
                            count += 1
                        assert orc.out_extent(size, pad, dil, k, stride) == count, (size, pad, dil, k, stride)


# --- accumulation ------------------------------------------------------------

def _im2col_acc(x, f, shape):
    """Explicit im2col of the zero-padded input, then an int64 matrix product."""
    N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw = shape
    xp = np.pad(x.astype(np.int64), ((0, 0), (0, 0), (ph, ph), (pw, pw)))
    Hp, Wp = xp.shape[2], xp.shape[3]
    P = 0
    while P * sh + dh * (R - 1) < Hp:
        P += 1
    Q = 0
    while Q * sw + dw * (S - 1) < Wp:
        Q += 1
    cols = np.zeros((N, P, Q, C, R, S), dtype=np.int64)
    for r in range(R):
        for s in range(S):
            win = xp[:, :, r * dh: r * dh + sh * (P - 1) + 1: sh, s * dw: s * dw + sw * (Q - 1) + 1: sw]
            cols[:, :, :, :, r, s] = win.transpose(0, 2, 3, 1)
    a = cols.reshape(N * P * Q, C * R * S)
    b = f.astype(np.int64).reshape(K, C * R * S)
    out = a @ b.T                                  # (N*P*Q, K)
    return out.reshape(N, P, Q, K).transpose(0, 3, 1, 2)


def _small_shapes(rng, count):
    shapes = []
    for i in range(count):
        N = int(rng.integers(1, 3))
        C = int(rng.integers(1, 5))
        H = int(rng.integers(3, 11))
        W = int(rng.integers(3, 11))
        K = int(rng.integers(1, 4))
        R = int(rng.integers(1, 4))
        S = int(rng.integers(1, 5))
        ph, pw = int(rng.integers(0, 3)), int(rng.integers(0, 3))
        sh, sw = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        dh, dw = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        if H + 2 * ph - dh * (R - 1) - 1 < 0 or W + 2 * pw - dw * (S - 1) - 1 < 0:
            continue
        shapes.append((N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw))
    return shapes


def pin_bruteforce_im2col(orc):
    """Random tiny shapes with every stride/pad/dilation in {1,2,3}-ish and
    R != S, H != W: the oracle equals explicit im2col + matrix product."""
    rng = np.random.default_rng(7)
    shapes = _small_shapes(rng, 60)
    # plus every (stride, dilation) pair on one fixed asymmetric shape
    for sh in (1, 2, 3):
        for sw in (1, 2, 3):
            for dh in (1, 2, 3):
                for dw in (1, 2, 3):
                    shapes.append((1, 2, 9, 11, 2, 2, 3, 1, 2, sh, sw, dh, dw))
    for shape in shapes:
        N, C, H, W, K, R, S = shape[:7]
        x = rng.integers(-128, 128, size=(N, C, H, W), dtype=np.int64).astype(np.int8)
        f = rng.integers(-128, 128, size=(K, C, R, S), dtype=np.int64).astype(np.int8)
        got = orc.conv_acc(x, f, shape, threads=2)
        want = _im2col_acc(x, f, shape)
        assert got.shape == want.shape, (shape, got.shape, want.shape)
        assert np.array_equal(got, want), shape


def pin_torch_conv2d_float64(orc):
    """Special case that reduces to a library routine: PyTorch's CPU conv2d in
    float64 on integer data is exact while sums stay below 2^53."""
    import torch
    rng = np.random.default_rng(11)
    shapes = [(2, 32, 12, 10, 32, 3, 3, 1, 1, 1, 1, 1, 1),
              (1, 32, 13, 17, 32, 3, 3, 1, 1, 2, 2, 1, 1),
              (1, 32, 20, 30, 4, 5, 9, 2, 4, 1, 1, 2, 3),
              (2, 64, 9, 9, 8, 3, 2, 0, 1, 2, 1, 1, 2)]
    for shape in shapes:
        N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw = shape
        x = rng.integers(-128, 128, size=(N, C, H, W), dtype=np.int64).astype(np.int8)
        f = rng.integers(-128, 128, size=(K, C, R, S), dtype=np.int64).astype(np.int8)
        want = torch.nn.functional.conv2d(
            torch.from_numpy(x.astype(np.float64)), torch.from_numpy(f.astype(np.float64)),
            stride=(sh, sw), padding=(ph, pw), dilation=(dh, dw)).numpy()
        got = orc.conv_acc(x, f, shape, threads=2)
        assert got.shape == want.shape
        assert np.array_equal(got.astype(np.float64), want), shape


def pin_all_ones_closed_form(orc):
    """All-ones tensors: acc = C * (#valid filter rows) * (#valid filter columns),
    the counts taken over taps that land inside the image."""
    cases = [(1, 3, 7, 9, 2, 3, 5, 1, 2, 1, 2, 2, 1),
             (2, 5, 6, 6, 1, 4, 2, 2, 0, 2, 1, 1, 3),
             (1, 32, 10, 12, 1, 5, 9, 2, 4, 1, 1, 2, 3),
             (1, 1, 5, 8, 1, 3, 3, 0, 1, 1, 3, 1, 1)]
    for shape in cases:
        N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw = shape
        x = np.ones((N, C, H, W), np.int8)
        f = np.ones((K, C, R, S), np.int8)
        acc = orc.conv_acc(x, f, shape, threads=1)
        P, Q = acc.shape[2], acc.shape[3]
        for p in range(P):
            rows = sum(1 for r in range(R) if ph <= p * sh + r * dh < ph + H)
            for q in range(Q):
                cols = sum(1 for s in range(S) if pw <= q * sw + s * dw < pw + W)
                assert np.all(acc[:, :, p, q] == C * rows * cols), (shape, p, q)


def pin_page4_interior_and_trace(orc):
    """Page 4's interior box and border count for its 512x512 dilated layer,
    and its hand trace of output[0,0,0,0], on all-ones data (one filter)."""
    g = _page4()
    d = dict(g["shape"])
    d["N"], d["K"] = 1, 1
    shape = _shape_of(d)
    C, R, S = d["C"], d["R"], d["S"]
    x = np.ones((1, C, d["H"], d["W"]), np.int8)
    f = np.ones((1, C, R, S), np.int8)
    acc = orc.conv_acc(x, f, shape)[0, 0]
    full = acc == C * R * S
    it = g["interior"]
    assert int(full.sum()) == it["interior_pixels"]
    assert int((~full).sum()) == it["border_pixels"]
    rows = np.nonzero(full.any(axis=1))[0]
    cols = np.nonzero(full.any(axis=0))[0]
    assert (rows.min(), rows.max(), cols.min(), cols.max()) == (it["oh_min"], it["oh_max"], it["ow_min"], it["ow_max"])
    assert np.all(full[it["oh_min"]:it["oh_max"] + 1, it["ow_min"]:it["ow_max"] + 1])
    tr = g["trace_output_0000"]
    rows_in = R - len(tr["rows_out_of_bounds"])                  # kh = 1..4 land inside
    cols_in = S - tr["row1_columns_in_bounds_from"]              # kw = 2..8 land inside
    assert acc[0, 0] == C * rows_in * cols_in


def pin_flop_count_page4(orc):
    """Page 4 counts about 371 GFLOP for its layer (2 ops per multiply-add)."""
    g = _page4()
    d = g["shape"]
    P, Q = orc.out_size(_shape_of(d))
    ops = 2 * d["N"] * d["K"] * P * Q * d["C"] * d["R"] * d["S"]
    assert abs(ops / 1e9 - g["total_gflop"]["value"]) <= g["total_gflop"]["relative_tolerance"] * g["total_gflop"]["value"]
    gv = g["gemm_view"]
    assert (d["K"], d["N"] * P * Q, d["C"] * d["R"] * d["S"]) == (gv["M_out_channels"], gv["N_pixels"], gv["K_reduction"])


# --- epilogue ----------------------------------------------------------------

def pin_epilogue_ties_half_even(orc):
    """alpha = 1/512 makes acc = 256 (mod 512) an exact .5: rint goes to even."""
    acc = np.array([256, 768, -256, -768, 1280, 255, 257, -257, 0, 512], np.int64)
    want = np.array([0, 2, 0, -2, 2, 0, 1, -1, 0, 1], np.int8)
    assert np.array_equal(orc.requantize(acc, 2.0 ** -9), want)


def pin_epilogue_saturation(orc):
    """Out-of-range results saturate to 127 / -128 (clamp to int8)."""
    shape = (1, 32, 4, 4, 2, 3, 3, 1, 1, 1, 1, 1, 1)
    x = np.full((1, 32, 4, 4), 127, np.int8)
    f = np.full((2, 32, 3, 3), 127, np.int8)
    acc = orc.conv_acc(x, f, shape)
    assert np.all(orc.requantize(acc, 1.0) == 127)
    x = np.full((1, 32, 4, 4), -128, np.int8)
    acc = orc.conv_acc(x, f, shape)
    assert np.all(orc.requantize(acc, 1.0) == -128)
    acc = np.array([2**31 - 1, -2**31, 1000, -1000, 128, -129, 127, -128], np.int64)
    assert np.array_equal(orc.requantize(acc, 1.0), np.array([127, -128, 127, -128, 127, -128, 127, -128], np.int8))
    assert np.array_equal(orc.requantize(np.array([3, -3], np.int64), 1e30), np.array([127, -128], np.int8))


def pin_epilogue_matches_ieee_single(orc):
    """The fp32 path against numpy's IEEE single multiply and half-even rint:
    int32 -> float32 (nearest even), one float32 multiply, rint, clamp."""
    rng = np.random.default_rng(3)
    acc = np.concatenate([rng.integers(-2**31, 2**31, 4000, dtype=np.int64),
                          rng.integers(-2**20, 2**20, 4000, dtype=np.int64),
                          rng.integers(-3000, 3000, 4000, dtype=np.int64)])
    for alpha in (2.0 ** -9, 2.0 ** -13, 0.3, 1.0 / 3.0, 7.25e-4, 1.0):
        a32 = np.float32(alpha)
        prod = acc.astype(np.int32).astype(np.float32) * a32
        want = np.clip(np.rint(prod), -128, 127).astype(np.int8)
        assert np.array_equal(orc.requantize(acc, alpha), want), alpha
    # power-of-two alphas: the single-precision product is exact, so the
    # result also equals the exact rational rounded half-even in float64.
    small = rng.integers(-2**24, 2**24 + 1, 4000, dtype=np.int64)
    for k in (9, 11, 12, 13, 18):
        want = np.clip(np.rint(small.astype(np.float64) * 2.0 ** -k), -128, 127).astype(np.int8)
        assert np.array_equal(orc.requantize(small, 2.0 ** -k), want), k


def pin_epilogue_float_conversion_rounds(orc):
    """(float)acc rounds to nearest even before the multiply: 5*2^22 + 1 is a
    tie between 5*2^22 and 5*2^22 + 2 and goes to 5*2^22, so with
    alpha = 2^-23 the product is exactly 2.5 and rint gives 2 (the exact
    rational 2.50000012 would give 3)."""
    acc = np.array([5 * 2**22 + 1, -(5 * 2**22 + 1)], np.int64)
    assert np.array_equal(orc.requantize(acc, 2.0 ** -23), np.array([2, -2], np.int8))


def pin_epilogue_int32_guard(orc):
    """Accumulators outside int32 are refused (the accumulator is int32)."""
    for bad in (2**31, -2**31 - 1):
        try:
            orc.requantize(np.array([bad], np.int64), 1.0)
        except OverflowError:
            continue
        raise AssertionError("int32 overflow not detected")


# --- per-output-channel epilogue: scale, bias, ReLU --------------------------

def pin_channel_epilogue_hand_values(orc):
    """clamp(rint(relu(alpha_k*acc + bias_k))) worked by hand: alpha_k =
    (0.5, 0.25, 2), bias_k = (0, -30.5, 1.5); every product and sum below is
    exact in fp32, and the .5 cases round half to even."""
    acc = np.array([[[3, 5, -7, 1000], [100, 142, 0, -1000], [10, -1, 63, -64]],
                    [[-3, 1, 255, -255], [122, 123, 126, -2], [0, 1, -2, 20]]], np.int64)
    alpha_k = np.array([0.5, 0.25, 2.0], np.float32)
    bias_k = np.array([0.0, -30.5, 1.5], np.float32)
    # n=0: 1.5->2, 2.5->2, -3.5->-4, 500->127 | 25-30.5=-5.5->-6, 35.5-30.5=5, -30.5->-30, -280.5->-128
    #      20+1.5=21.5->22, -2+1.5=-0.5->0, 127.5->127, -126.5->-126
    # n=1: -1.5->-2, 0.5->0, 127.5->127, -127.5->-128 | 0, 0.25->0, 1, -31
    #      1.5->2, 3.5->4, -2.5->-2, 41.5->42
    want = np.array([[[2, 2, -4, 127], [-6, 5, -30, -128], [22, 0, 127, -126]],
                     [[-2, 0, 127, -128], [0, 0, 1, -31], [2, 4, -2, 42]]], np.int8)
    want_relu = np.array([[[2, 2, 0, 127], [0, 5, 0, 0], [22, 0, 127, 0]],
                          [[0, 0, 127, 0], [0, 0, 1, 0], [2, 4, 0, 42]]], np.int8)
    assert np.array_equal(orc.requantize_channels(acc, 1.0, alpha_k, bias_k, relu=False), want)
    assert np.array_equal(orc.requantize_channels(acc, 1.0, alpha_k, bias_k, relu=True), want_relu)
    # no bias: the scale alone; no per-channel scale: the scalar alpha
    assert np.array_equal(orc.requantize_channels(acc[:, :1], 1.0, alpha_k[:1]), np.array([[[2, 2, -4, 127]], [[-2, 0, 127, -128]]], np.int8))
    assert np.array_equal(orc.requantize_channels(acc[:, 1:2], 0.25, None, bias_k[1:2]), np.array([[[-6, 5, -30, -128]], [[0, 0, 1, -31]]], np.int8))


def pin_channel_epilogue_separate_roundings(orc):
    """One fp32 multiply, then one fp32 add, each rounded: alpha = fp32(1/3) =
    11184811 * 2^-25 and acc = 6 give the exact product 2 + 2^-24, which
    rounds to 2.0 (a quarter of an ulp above it); 2.0 - 1.5 = 0.5 and rint
    gives 0.  A fused multiply-add would keep 0.5 + 2^-24 (representable)
    and give 1."""
    acc = np.array([[[6]]], np.int64)
    y = orc.requantize_channels(acc, 1.0, np.array([1.0 / 3.0], np.float32), np.array([-1.5], np.float32))
    assert y.reshape(-1)[0] == 0


def pin_channel_epilogue_reduces_to_alpha_only(orc):
    """Equal scales, no bias, no ReLU: the alpha-only clamp epilogue."""
    rng = np.random.default_rng(17)
    acc = rng.integers(-2**31, 2**31, (3, 4, 50), dtype=np.int64)
    for alpha in (2.0 ** -9, 0.3, 1.0 / 3.0):
        ak = np.full(4, alpha, np.float32)
        assert np.array_equal(orc.requantize_channels(acc, 5.0, ak), orc.requantize(acc, alpha).reshape(acc.shape))
        assert np.array_equal(orc.requantize_channels(acc, alpha), orc.requantize(acc, alpha).reshape(acc.shape))


# --- fp32 direct convolution (page 4's nn.Conv2d), evaluated in double -------

_F32_SHAPES = [(2, 3, 9, 11, 4, 3, 5, 1, 2, 1, 1, 1, 1),
               (1, 2, 12, 30, 3, 5, 9, 2, 4, 1, 1, 2, 3),
               (2, 4, 13, 9, 2, 3, 3, 1, 0, 2, 3, 1, 2),
               (1, 5, 8, 8, 3, 2, 3, 0, 1, 3, 2, 3, 1)]


def pin_f64_integer_data_matches_int_accumulators(orc):
    """On integer-valued inputs every product and partial sum is an exact
    integer in double, so y must equal the integer path's accumulators (which
    are pinned to im2col, PyTorch and closed forms above) plus the bias."""
    rng = np.random.default_rng(23)
    for shape in _F32_SHAPES:
        N, C, H, W, K, R, S = shape[:7]
        x = rng.integers(-128, 128, size=(N, C, H, W)).astype(np.int8)
        f = rng.integers(-128, 128, size=(K, C, R, S)).astype(np.int8)
        b = rng.integers(-1000, 1000, size=K).astype(np.float32)
        y, mag = orc.conv_f64(x.astype(np.float32), f.astype(np.float32), shape, bias=b, threads=2)
        acc = orc.conv_acc(x, f, shape, threads=2)
        assert np.array_equal(y, acc.astype(np.float64) + b.astype(np.float64)[None, :, None, None]), shape
        assert np.all(mag >= np.abs(y))


def pin_f64_matches_torch_conv2d(orc):
    """Random fp32 data: PyTorch's CPU conv2d in float64 with bias agrees to
    within double rounding of the magnitude sum."""
    import torch
    rng = np.random.default_rng(29)
    for shape in _F32_SHAPES:
        N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw = shape
        x = rng.random((N, C, H, W)).astype(np.float32)
        w = (rng.random((K, C, R, S)) * 2 - 1).astype(np.float32)
        b = (rng.random(K) * 2 - 1).astype(np.float32)
        want = torch.nn.functional.conv2d(torch.from_numpy(x.astype(np.float64)), torch.from_numpy(w.astype(np.float64)),
                                          torch.from_numpy(b.astype(np.float64)), stride=(sh, sw), padding=(ph, pw),
                                          dilation=(dh, dw)).numpy()
        y, mag = orc.conv_f64(x, w, shape, bias=b, threads=2)
        assert y.shape == want.shape, shape
        assert np.all(np.abs(y - want) <= 1e-13 * mag + 1e-300), shape


def pin_f64_bias_only_and_magnitudes(orc):
    """Zero input: every output is its channel's bias and the magnitude is
    |bias|.  Non-negative data: the magnitude sum equals the output."""
    shape = (2, 3, 7, 6, 4, 3, 2, 1, 0, 1, 2, 2, 1)
    N, C, H, W, K, R, S = shape[:7]
    b = np.array([0.5, -1.25, 3.0, -0.0625], np.float32)
    y, mag = orc.conv_f64(np.zeros((N, C, H, W), np.float32), np.ones((K, C, R, S), np.float32), shape, bias=b)
    assert np.array_equal(y, np.broadcast_to(b.astype(np.float64)[None, :, None, None], y.shape))
    assert np.array_equal(mag, np.abs(y))
    rng = np.random.default_rng(31)
    x = rng.random((N, C, H, W)).astype(np.float32)
    w = rng.random((K, C, R, S)).astype(np.float32)
    y, mag = orc.conv_f64(x, w, shape, bias=np.abs(b))
    assert np.array_equal(y, mag)


def pin_f64_page4_trace(orc):
    """Page 4's hand trace of output[0,0,0,0] for its 5x9 dilated layer on
    all-ones data: 4 in-bounds filter rows x 7 in-bounds columns x 32
    channels, plus the bias."""
    g = _page4()
    d = dict(g["shape"])
    d["N"], d["K"], d["H"], d["W"] = 1, 1, 40, 40
    shape = _shape_of(d)
    C, R, S = d["C"], d["R"], d["S"]
    tr = g["trace_output_0000"]
    rows_in = R - len(tr["rows_out_of_bounds"])
    cols_in = S - tr["row1_columns_in_bounds_from"]
    y, _ = orc.conv_f64_points(np.ones((1, C, 40, 40), np.float32), np.ones((1, C, R, S), np.float32), shape,
                               np.array([[0, 0, 0, 0]]), bias=np.array([0.5], np.float32))
    assert y[0] == C * rows_in * cols_in + 0.5


def pin_f32_error_bound_worked_values(orc):
    """gamma_n = n*u/(1 - n*u) with u = 2^-24, worked by hand: one product plus
    the bias (n = 2) gives 2^-23/(1 - 2^-23) = 1/(2^23 - 1) = 1/8388607; two
    products plus the bias (n = 3) give 3*2^-24/(1 - 3*2^-24) = 3/16777213."""
    assert orc.f32_error_bound(1.0, 1) == 1.0 / 8388607.0
    assert orc.f32_error_bound(1.0, 2) == 3.0 / 16777213.0
    assert orc.f32_error_bound(0.0, 1440) == 0.0


def pin_f32_error_bound_attained(orc):
    """The bound is nearly attained, so it cannot be loose by a constant
    factor: summing 1 and then m addends of 2^-24 in single precision loses
    every addend (1 + 2^-24 lies halfway between 1 and its successor 1 + 2^-23
    and ties to the even 1), an error of m*2^-24 on m + 1 summands of
    magnitude 1 + m*2^-24, while gamma_{m+1} times that magnitude is only
    (m+1)/m times as large, to first order in u."""
    for m in (1, 7, 100):
        s = np.float32(0.0)
        for v in [np.float32(1.0)] + [np.float32(2.0 ** -24)] * m:
            s = np.float32(s + v)
        assert s == np.float32(1.0)
        exact = 1.0 + m * 2.0 ** -24
        err = exact - float(s)
        bound = float(orc.f32_error_bound(exact, m))   # m products plus the bias: m + 1 summands
        assert err <= bound, (m, err, bound)
        assert err >= bound * m / (m + 1) * (1.0 - 1e-4), (m, err, bound)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
