"""The no-allocation entry point, i8c_conv2d_fprop_noalloc.

Some callers cannot let a library call cudaMalloc: their device memory is
owned by a framework allocator or a fixed pool, or they run on a path where
the allocator's implicit synchronisation is not allowed.  For them the
library offers a variant whose scratch lives in a fixed static device array.
These tests call it through the C-ABI and check that it produces exactly
what the oracle and the regular checked entry point produce (the convolution
is bit-exact, so the tolerance is zero): on two calls in a row that reuse the
shared scratch with different filters and shapes, on the largest filter the
scratch holds, and after a bounded wait that ran out (which the status query
reports).  The file is collected last so
that a run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


def _device_inputs(torch, shape, seed):
    N, C, H, W, K, R, S = shape[:7]
    x = synth.uniform_int8(seed, N * C * H * W, -128, 127).reshape(N, C, H, W)
    f = synth.uniform_int8(seed + 1, K * C * R * S, -128, 127).reshape(K, C, R, S)
    xd = torch.from_numpy(oracle.nchw_to_ncxhwx32(x)).cuda()
    fd = torch.from_numpy(oracle.kcrs_to_cxrskx32(f)).cuda()
    return xd, fd


def _noalloc(ext, xd, fd, yd, shape, alpha, stream):
    return ext.lib.i8c_conv2d_fprop_noalloc(xd.data_ptr(), fd.data_ptr(), yd.data_ptr(),
                                            ctypes.byref(ext.ConvShape.of(shape)), ctypes.c_float(alpha),
                                            stream.cuda_stream)


def _oracle_packed_y(shape, seed, alpha):
    N, C, H, W, K, R, S = shape[:7]
    x = synth.uniform_int8(seed, N * C * H * W, -128, 127).reshape(N, C, H, W)
    f = synth.uniform_int8(seed + 1, K * C * R * S, -128, 127).reshape(K, C, R, S)
    y, _ = oracle.Oracle().conv2d_fprop(x, f, shape, alpha)
    return oracle.nchw_to_ncxhwx32(y).reshape(-1)


def test_noalloc_matches_oracle_and_checked_entry_point_on_two_calls():
    import torch
    import int8_implicit_gemm_gb300 as ext
    stream = torch.cuda.current_stream()
    cases = [
        ((4, 256, 20, 20, 256, 3, 3, 1, 1, 1, 1, 1, 1), 2.0 ** -12, 31),   # larger filter first
        ((2, 64, 17, 15, 96, 5, 3, 2, 1, 2, 1, 1, 2), 2.0 ** -10, 57),     # then a smaller one
    ]
    runs = []
    for shape, alpha, seed in cases:
        xd, fd = _device_inputs(torch, shape, seed)
        P, Q = ext.i8c_output_size(shape)
        y = torch.full((shape[0] * shape[4] * P * Q,), 99, dtype=torch.int8, device="cuda")
        runs.append((shape, alpha, seed, xd, fd, y))
    # two no-allocation calls back to back on one stream
    for shape, alpha, _, xd, fd, y in runs:
        assert _noalloc(ext, xd, fd, y, shape, alpha, stream) == ext.I8C_OK
    assert ext.i8c_last_device_status(stream) == ext.I8C_OK
    # the regular checked entry point on the same inputs
    refs = []
    for shape, alpha, _, xd, fd, y in runs:
        y_ref = torch.empty_like(y)
        ext.i8c_conv2d_fprop(xd, fd, y_ref, shape, alpha, stream)
        refs.append(y_ref)
    torch.cuda.synchronize()
    for (shape, alpha, seed, _, _, y), y_ref in zip(runs, refs):
        got = y.cpu().numpy()
        assert np.array_equal(got, y_ref.cpu().numpy()), shape
        assert np.array_equal(got, _oracle_packed_y(shape, seed, alpha)), shape


def test_noalloc_largest_filter_that_fits():
    """The largest filter the fixed array holds (K*C*R*S = 4,193,280 of at
    most 4,194,176 elements): its fp16 copy and the filter tensor map reach
    the array's last bytes.  Exact against the oracle and the checked entry
    point."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    shape, alpha, seed = (1, 1120, 6, 6, 416, 3, 3, 1, 1, 1, 1, 1, 1), 2.0 ** -13, 91
    assert ext.i8c_supported(shape) == ext.I8C_OK
    stream = torch.cuda.current_stream()
    xd, fd = _device_inputs(torch, shape, seed)
    P, Q = ext.i8c_output_size(shape)
    y = torch.full((shape[0] * shape[4] * P * Q,), 99, dtype=torch.int8, device="cuda")
    assert _noalloc(ext, xd, fd, y, shape, alpha, stream) == ext.I8C_OK
    y_ref = torch.empty_like(y)
    ext.i8c_conv2d_fprop(xd, fd, y_ref, shape, alpha, stream)
    assert ext.i8c_last_device_status(stream) == ext.I8C_OK
    got = y.cpu().numpy()
    assert np.array_equal(got, y_ref.cpu().numpy())
    assert np.array_equal(got, _oracle_packed_y(shape, seed, alpha))


def test_noalloc_timeout_is_reported():
    """A bounded wait that runs out inside the no-allocation call (a producer
    skips one arrival on purpose, through the test hook) is reported by
    i8c_last_device_status, once; the next call is exact again."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    shape, alpha, seed = (2, 64, 16, 16, 64, 3, 3, 1, 1, 1, 1, 1, 1), 2.0 ** -10, 71
    stream = torch.cuda.current_stream()
    xd, fd = _device_inputs(torch, shape, seed)
    y = torch.zeros(2 * 64 * 256, dtype=torch.int8, device="cuda")
    try:
        ext.i8c_debug_set_oneshot(ext.I8C_DEBUG_SKIP_FIRST_ARRIVE, 20000)
        assert _noalloc(ext, xd, fd, y, shape, alpha, stream) == ext.I8C_OK
        assert ext.i8c_last_device_status(stream) == ext.I8C_ERR_TIMEOUT
        assert ext.i8c_last_device_status(stream) == ext.I8C_OK
    finally:
        ext.i8c_debug_set_oneshot(0, 0)
    assert _noalloc(ext, xd, fd, y, shape, alpha, stream) == ext.I8C_OK
    assert ext.i8c_last_device_status(stream) == ext.I8C_OK
    assert np.array_equal(y.cpu().numpy(), _oracle_packed_y(shape, seed, alpha))


def test_noalloc_rejects_filter_beyond_scratch():
    import torch
    import int8_implicit_gemm_gb300 as ext
    shape = (1, 1024, 8, 8, 512, 3, 3, 1, 1, 1, 1, 1, 1)   # 4,718,592 filter elements > 4,194,176
    assert ext.i8c_supported(shape) == ext.I8C_OK
    buf = torch.zeros(64, dtype=torch.int8, device="cuda")
    st = _noalloc(ext, buf, buf, buf, shape, 1.0, torch.cuda.current_stream())
    assert st == ext.I8C_ERR_UNSUPPORTED
