"""GPU tests of the boundary itself: layout kernels, the one-shot entry
points, host-buffer runs, alignment errors and the bounded-wait failure path."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available()
    return torch


def test_pack_unpack_activations(torch_cuda):
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    N, C, H, W = 3, 96, 7, 5
    a = synth.uniform_int8(3, N * C * H * W, -128, 127).reshape(N, C, H, W)
    src = torch.from_numpy(a).cuda()
    dst = torch.empty_like(src)
    ext.i8c_pack_nchw_to_ncxhwx32(src, dst, N, C, H, W)
    assert np.array_equal(dst.cpu().numpy().reshape(-1), oracle.nchw_to_ncxhwx32(a).reshape(-1))
    back = torch.empty_like(src)
    ext.i8c_unpack_ncxhwx32_to_nchw(dst, back, N, C, H, W)
    assert np.array_equal(back.cpu().numpy(), a)


def test_pack_unpack_filters(torch_cuda):
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    K, C, R, S = 64, 64, 5, 3
    f = synth.uniform_int8(4, K * C * R * S, -128, 127).reshape(K, C, R, S)
    src = torch.from_numpy(f).cuda()
    dst = torch.empty_like(src)
    ext.i8c_pack_kcrs_to_cxrskx32(src, dst, K, C, R, S)
    assert np.array_equal(dst.cpu().numpy().reshape(-1), oracle.kcrs_to_cxrskx32(f).reshape(-1))
    back = torch.empty_like(src)
    ext.i8c_unpack_cxrskx32_to_kcrs(dst, back, K, C, R, S)
    assert np.array_equal(back.cpu().numpy(), f)


def test_one_shot_entry_points(torch_cuda):
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    shape = (2, 64, 20, 20, 128, 3, 3, 1, 1, 1, 1, 1, 1)
    x = synth.uniform_int8(10, 2 * 64 * 400, -128, 127).reshape(2, 64, 20, 20)
    f = synth.uniform_int8(11, 128 * 64 * 9, -128, 127).reshape(128, 64, 3, 3)
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -11)
    xp, fp = gpu_util.packed_inputs(x, f)
    xd, fd = torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda()
    y = ext.conv2d_fprop(xd, fd, shape, 2.0 ** -11)
    acc = torch.empty(y.shape, dtype=torch.int32, device="cuda")
    ext.i8c_conv2d_fprop_acc(xd, fd, acc, shape)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), y_ref)
    assert np.array_equal(acc.cpu().numpy(), acc_ref.astype(np.int32))


def test_host_buffer_run(torch_cuda):
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    shape = (2, 32, 24, 24, 64, 3, 3, 1, 1, 1, 1, 1, 1)
    x = synth.uniform_int8(12, 2 * 32 * 576, -128, 127).reshape(2, 32, 24, 24)
    f = synth.uniform_int8(13, 64 * 32 * 9, -128, 127).reshape(64, 32, 3, 3)
    y_ref, _ = gpu_util.oracle_packed(shape, x, f, 2.0 ** -9)
    xp, fp = gpu_util.packed_inputs(x, f)
    xh = torch.from_numpy(xp).pin_memory()
    fh = torch.from_numpy(fp).pin_memory()
    yh = torch.empty(y_ref.size, dtype=torch.int8).pin_memory()
    plan = ext.Plan(shape, host_staging=True)
    stream = torch.cuda.current_stream()
    plan.run_host(xh, fh, yh, 2.0 ** -9, stream)
    stream.synchronize()
    assert plan.status() == 0
    assert np.array_equal(yh.numpy(), y_ref.reshape(-1))


def test_host_buffer_pipelined_runs(torch_cuda):
    """i8c_plan_run_host_pipelined: five end-to-end runs on pinned host
    buffers with different inputs, alphas and outputs, the copies of
    neighbouring runs overlapped on the plan's copy streams: every output
    exact against the oracle once the caller's stream is synchronised."""
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    shape = (2, 64, 18, 18, 128, 3, 3, 1, 1, 1, 1, 1, 1)
    N, C, H, W, K = shape[:5]
    plan = ext.Plan(shape, host_staging=2)
    xs, fs, ys, alphas, refs = [], [], [], [], []
    for i in range(5):
        x = synth.uniform_int8(40 + i, N * C * H * W, -128, 127).reshape(N, C, H, W)
        f = synth.uniform_int8(50 + i, K * C * 9, -128, 127).reshape(K, C, 3, 3)
        alpha = 2.0 ** -(9 + i)
        y_ref, _ = gpu_util.oracle_packed(shape, x, f, alpha)
        xp, fp = gpu_util.packed_inputs(x, f)
        xs.append(torch.from_numpy(xp).pin_memory())
        fs.append(torch.from_numpy(fp).pin_memory())
        ys.append(torch.full((y_ref.size,), 77, dtype=torch.int8).pin_memory())
        alphas.append(alpha)
        refs.append(y_ref.reshape(-1))
    stream = torch.cuda.Stream()
    plan.run_host_pipelined(xs, fs, ys, alphas, stream)
    stream.synchronize()
    assert plan.status(stream) == 0
    for i in range(5):
        assert np.array_equal(ys[i].numpy(), refs[i]), i
    plan.destroy()
    with pytest.raises(ext.I8ConvError):      # a plan without the second staging set
        p1 = ext.Plan(shape, host_staging=1)
        try:
            p1.run_host_pipelined(xs[:1], fs[:1], ys[:1], alphas[:1], stream)
        finally:
            p1.destroy()


def test_misaligned_pointer_rejected(torch_cuda):
    import ctypes
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    shape = (1, 32, 8, 8, 32, 3, 3, 1, 1, 1, 1, 1, 1)
    x = torch.zeros(32 * 64 + 16, dtype=torch.int8, device="cuda")
    f = torch.zeros(32 * 32 * 9, dtype=torch.int8, device="cuda")
    y = torch.zeros(32 * 64, dtype=torch.int8, device="cuda")
    plan = ext.Plan(shape)
    st = ext.lib.i8c_plan_run(plan.handle, x.data_ptr() + 1, f.data_ptr(), y.data_ptr(), ctypes.c_float(1.0),
                              torch.cuda.current_stream().cuda_stream)
    assert st == ext.I8C_ERR_MISALIGNED


def test_bounded_wait_reports_timeout_and_context_survives(torch_cuda):
    """A producer skips one arrival on purpose: the MMA warp's wait runs out
    after 20 ms, every role stops, the kernel returns and the plan reports
    I8C_ERR_TIMEOUT (gather kernel, halo kernel, halo kernel on CTA pairs,
    transposed tiles, on single CTAs and on pairs, stacked taps; halos by
    registers and by TMA; resident filters written by the kernel itself and
    loaded by TMA from the conversion kernel's copy).
    The same context then runs a correct convolution."""
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    shape = (2, 64, 16, 16, 64, 3, 3, 1, 1, 1, 1, 1, 1)
    x = synth.uniform_int8(14, 2 * 64 * 256, -128, 127).reshape(2, 64, 16, 16)
    f = synth.uniform_int8(15, 64 * 64 * 9, -128, 127).reshape(64, 64, 3, 3)
    xp, fp = gpu_util.packed_inputs(x, f)
    xd, fd = torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda()
    y = torch.zeros(2 * 64 * 256, dtype=torch.int8, device="cuda")
    for kernel, loads, fused in ((1, 0, 0), (2, 0, 0), (3, 0, 0), (4, 0, 0), (5, 0, 0), (6, 0, 0), (2, 3, 0),
                                 (3, 3, 0), (4, 3, 0), (5, 3, 0), (2, 0, 2), (3, 0, 2), (3, 0, 3)):
        bad = ext.Plan(shape, wait_timeout_us=20000, debug_flags=ext.I8C_DEBUG_SKIP_FIRST_ARRIVE,
                       kernel_variant=kernel, halo_loads=loads, fused_filter=fused,
                       block_n=64 if fused == 2 else 0)  # one 64-channel tile: a resident filter
        bad.run(xd, fd, y, 1.0)
        assert bad.status() == ext.I8C_ERR_TIMEOUT, (kernel, loads, fused)
        assert bad.status() == ext.I8C_OK          # the status word was cleared
    y_ref, _ = gpu_util.oracle_packed(shape, x, f, 2.0 ** -10)
    y2, _ = gpu_util.gpu_run(shape, x, f, 2.0 ** -10, want_acc=False)
    assert np.array_equal(y2, y_ref)


def test_one_shot_timeout_reported_by_last_device_status(torch_cuda):
    """A bounded wait that runs out inside a checked one-shot call (a producer
    skips one arrival on purpose, through the one-shot test hook) surfaces as
    I8C_ERR_TIMEOUT from i8c_last_device_status on that call's stream, once;
    after the hook is removed the next one-shot call is bit-exact."""
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    shape = (2, 64, 16, 16, 64, 3, 3, 1, 1, 1, 1, 1, 1)
    x = synth.uniform_int8(16, 2 * 64 * 256, -128, 127).reshape(2, 64, 16, 16)
    f = synth.uniform_int8(17, 64 * 64 * 9, -128, 127).reshape(64, 64, 3, 3)
    xp, fp = gpu_util.packed_inputs(x, f)
    xd, fd = torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda()
    y = torch.zeros(2 * 64 * 256, dtype=torch.int8, device="cuda")
    acc = torch.zeros(2 * 64 * 256, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    try:
        ext.i8c_debug_set_oneshot(ext.I8C_DEBUG_SKIP_FIRST_ARRIVE, 20000)
        ext.i8c_conv2d_fprop(xd, fd, y, shape, 1.0, stream)
        assert ext.i8c_last_device_status(stream) == ext.I8C_ERR_TIMEOUT
        assert ext.i8c_last_device_status(stream) == ext.I8C_OK      # read once, then cleared
        ext.i8c_conv2d_fprop_acc(xd, fd, acc, shape, stream)
        assert ext.i8c_last_device_status(stream) == ext.I8C_ERR_TIMEOUT
    finally:
        ext.i8c_debug_set_oneshot(0, 0)
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -10)
    ext.i8c_conv2d_fprop(xd, fd, y, shape, 2.0 ** -10, stream)
    ext.i8c_conv2d_fprop_acc(xd, fd, acc, shape, stream)
    assert ext.i8c_last_device_status(stream) == ext.I8C_OK
    assert np.array_equal(y.cpu().numpy(), y_ref.reshape(-1))
    assert np.array_equal(acc.cpu().numpy(), acc_ref.astype(np.int32).reshape(-1))


def test_one_shot_plan_cache_is_bounded(torch_cuda):
    """A caller that keeps presenting new cache keys (a new shape or a new
    stream for every call) cannot grow the one-shot plan cache beyond its
    bound: the least recently used plan makes room, and every call stays
    exact.  (Shapes stand in for streams here: torch hands out its streams
    from a small pool, so new torch streams would repeat keys.)"""
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    stream = torch.cuda.current_stream()
    ext.i8c_debug_set_oneshot(0, 0)          # starts from an empty cache
    for i in range(70):
        shape = (1, 32, 6 + i % 10, 6 + i // 10, 32, 3, 3, 1, 1, 1, 1, 1, 1)
        N, C, H, W, K = shape[:5]
        x = synth.uniform_int8(18 + i, C * H * W, -128, 127).reshape(1, C, H, W)
        f = synth.uniform_int8(19, K * C * 9, -128, 127).reshape(K, C, 3, 3)
        y_ref, _ = gpu_util.oracle_packed(shape, x, f, 2.0 ** -9)
        xp, fp = gpu_util.packed_inputs(x, f)
        xd, fd = torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda()
        y = torch.zeros(y_ref.size, dtype=torch.int8, device="cuda")
        ext.i8c_conv2d_fprop(xd, fd, y, shape, 2.0 ** -9, stream)
        assert ext.i8c_last_device_status(stream) == ext.I8C_OK
        assert np.array_equal(y.cpu().numpy(), y_ref.reshape(-1)), i
        assert ext.i8c_oneshot_cached_plans() == min(i + 1, 64)
    ext.i8c_debug_set_oneshot(0, 0)
    assert ext.i8c_oneshot_cached_plans() == 0


@pytest.mark.parametrize("opts", [{}, dict(kernel_variant=1), dict(kernel_variant=2), dict(kernel_variant=3),
                                  dict(kernel_variant=4), dict(kernel_variant=5), dict(kernel_variant=6)],
                         ids=["auto", "gather", "halo", "halo-pair", "transposed", "transposed-pair", "stacked"])
def test_host_layout_matches_real_plans(torch_cuda, opts):
    """The layout the host-only planner reports (the one the CPU bounds check
    inspects) is the layout real plans give their kernels on this GPU."""
    import int8_implicit_gemm_gb300 as ext
    sms = torch_cuda.cuda.get_device_properties(0).multi_processor_count
    for wl in synth.WORKLOADS:
        shape = wl.shape_tuple()
        try:
            plan = ext.Plan(shape, **opts)
        except ext.I8ConvError as e:
            assert e.status == ext.I8C_ERR_UNSUPPORTED
            continue
        assert plan.layout() == ext.i8c_plan_layout(shape, sms, **opts), wl.name
        plan.destroy()


def test_plan_runs_captured_in_a_cuda_graph(torch_cuda):
    """i8c_plan_run is capturable: a CUDA graph of three runs on different
    inputs replays to the oracle's outputs (the dependent launch of the
    convolution after the filter conversion becomes a graph edge)."""
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    shape = (2, 64, 13, 11, 64, 3, 3, 1, 1, 1, 1, 1, 1)
    plan = ext.Plan(shape)
    P, Q = plan.info["P"], plan.info["Q"]
    cases = []
    for seed in (31, 32, 33):
        x = synth.uniform_int8(seed, 2 * 64 * 13 * 11, -128, 127).reshape(2, 64, 13, 11)
        f = synth.uniform_int8(seed + 100, 64 * 64 * 9, -128, 127).reshape(64, 64, 3, 3)
        xp, fp = gpu_util.packed_inputs(x, f)
        y = torch.zeros(2 * 64 * P * Q, dtype=torch.int8, device="cuda")
        cases.append((x, f, torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda(), y))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.run(cases[0][2], cases[0][3], cases[0][4], 2.0 ** -10, s)  # warm-up outside the graph
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _, _, xd, fd, y in cases:
            plan.run(xd, fd, y, 2.0 ** -10, torch.cuda.current_stream())
    for _, _, _, _, y in cases:
        y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert plan.status() == ext.I8C_OK
    for x, f, _, _, y in cases:
        y_ref, _ = gpu_util.oracle_packed(shape, x, f, 2.0 ** -10)
        assert np.array_equal(y.cpu().numpy().reshape(y_ref.shape), y_ref)
    plan.destroy()


def test_filter_conversion_inside_the_kernel(torch_cuda):
    """fused_filter = 1: the halo kernel converts the filter itself behind a
    grid barrier (one launch per run); outputs stay exact over repeated runs
    with different filters."""
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    shape = (2, 64, 13, 11, 256, 3, 3, 1, 1, 1, 1, 1, 1)
    plan = ext.Plan(shape, kernel_variant=2, fused_filter=1)
    assert plan.info["kernels_per_run"] == 1
    P, Q = plan.info["P"], plan.info["Q"]
    for seed in (41, 42, 43):
        x = synth.uniform_int8(seed, 2 * 64 * 13 * 11, -128, 127).reshape(2, 64, 13, 11)
        f = synth.uniform_int8(seed + 7, 256 * 64 * 9, -128, 127).reshape(256, 64, 3, 3)
        xp, fp = gpu_util.packed_inputs(x, f)
        y = torch.zeros(2 * 256 * P * Q, dtype=torch.int8, device="cuda")
        plan.run(torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda(), y, 2.0 ** -11)
        torch.cuda.synchronize()
        assert plan.status() == ext.I8C_OK
        y_ref, _ = gpu_util.oracle_packed(shape, x, f, 2.0 ** -11)
        assert np.array_equal(y.cpu().numpy().reshape(y_ref.shape), y_ref)
    plan.destroy()


def test_channel_epilogue_misaligned_rejected(torch_cuda):
    """Per-channel scale or bias arrays must be 16-byte aligned (the kernels
    read them with vector loads): a 4-byte offset is refused before launch."""
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    shape = (1, 32, 8, 8, 32, 3, 3, 1, 1, 1, 1, 1, 1)
    plan = ext.Plan(shape)
    x = torch.zeros(32 * 64, dtype=torch.int8, device="cuda")
    f = torch.zeros(32 * 32 * 9, dtype=torch.int8, device="cuda")
    y = torch.zeros(32 * 64, dtype=torch.int8, device="cuda")
    ones = torch.ones(40, dtype=torch.float32, device="cuda")
    for kw in (dict(alpha_k=ones[1:33]), dict(bias=ones[1:33])):
        with pytest.raises(ext.I8ConvError) as ei:
            plan.run(x, f, y, 1.0, **kw)
        assert ei.value.status == ext.I8C_ERR_MISALIGNED
    plan.run(x, f, y, 1.0, alpha_k=ones[:32], bias=ones[4:36], relu=True)
    assert plan.status() == ext.I8C_OK
    plan.destroy()


@pytest.mark.parametrize("shape", [(2, 64, 20, 20, 128, 3, 3, 1, 1, 1, 1, 1, 1),
                                   (1, 64, 23, 23, 64, 3, 3, 1, 1, 2, 2, 1, 1)], ids=["stride1", "stride2"])
def test_autotune_picks_an_exact_plan(torch_cuda, shape):
    """The tuner times every candidate that the shape supports, returns the
    fastest, leaves that plan's (bit-exact) output in y, and its options give
    a plan whose output is bit-exact too."""
    import int8_implicit_gemm_gb300 as ext
    torch = torch_cuda
    N, C, H, W, K, R, S = shape[:7]
    x = synth.uniform_int8(40, N * C * H * W, -128, 127).reshape(N, C, H, W)
    f = synth.uniform_int8(41, K * C * R * S, -128, 127).reshape(K, C, R, S)
    alpha = 2.0 ** -11
    y_ref, _ = gpu_util.oracle_packed(shape, x, f, alpha)
    xp, fp = gpu_util.packed_inputs(x, f)
    xd, fd = torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda()
    y = torch.full(y_ref.shape, 77, dtype=torch.int8, device="cuda")
    best, best_us, entries = ext.i8c_plan_autotune(xd, fd, y, shape, alpha, iters=3)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), y_ref)
    ok = [e for e in entries if e[1] == 0]
    assert entries[0][0]["kernel_variant"] == 0 and entries[0][1] == 0      # the default runs first
    assert len(ok) >= 3 and all(e[2] > 0 for e in ok)
    assert best_us == pytest.approx(min(e[2] for e in ok))
    assert best in [e[0] for e in ok]
    if shape[9] == 2:  # transposed tiles are stride-1 only
        assert all(e[1] == ext.I8C_ERR_UNSUPPORTED for e in entries if e[0]["kernel_variant"] in (4, 5))
    plan = ext.Plan(shape, **best)
    y2 = torch.empty_like(y)
    plan.run(xd, fd, y2, alpha)
    torch.cuda.synchronize()
    assert plan.status() == 0
    assert np.array_equal(y2.cpu().numpy(), y_ref)
    plan.destroy()
