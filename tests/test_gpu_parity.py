"""GPU parity: the tcgen05 implicit-GEMM path against the CPU oracle, bit for
bit, on seeded inputs -- int32 accumulators and int8 outputs, element by
element: small shapes that span several tiles and ragged tails, and the five
full-size workloads in full."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util

pytestmark = pytest.mark.gpu

SMALL = [
    # N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw
    (1, 32, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1),     # the 16x16 single-image layer, two tiles
    (2, 64, 13, 11, 64, 3, 3, 1, 1, 1, 1, 1, 1),     # ragged last tile (286 rows)
    (3, 32, 30, 30, 96, 5, 9, 2, 4, 1, 1, 2, 3),     # dilated 5x9, K=96 inside a 128-wide tile
    (2, 128, 23, 23, 256, 3, 3, 1, 1, 2, 2, 1, 1),   # stride 2, two exact-fp32 chunks
    (1, 64, 12, 12, 512, 3, 3, 1, 1, 1, 1, 1, 1),    # two N-tiles of 256
    (1, 512, 6, 6, 64, 3, 3, 1, 1, 1, 1, 1, 1),      # 4608-long reduction, five chunks
    (4, 64, 10, 10, 32, 1, 1, 0, 0, 1, 1, 1, 1),     # 1x1 filter
    (2, 32, 17, 19, 64, 3, 2, 2, 1, 3, 2, 2, 3),     # mixed stride / dilation / padding per axis
    (2, 32, 3, 3, 32, 3, 3, 0, 0, 1, 1, 1, 1),       # 1x1 output
    (1, 32, 1, 1, 32, 3, 3, 1, 1, 1, 1, 1, 1),       # 1x1 input, all but the centre tap padded
    (5, 96, 9, 7, 160, 2, 3, 0, 1, 1, 2, 2, 1),      # K=160 -> 256-wide tile, C=96
]


def _data(shape, seed, lo=-128, hi=127):
    N, C, H, W, K, R, S = shape[:7]
    x = synth.uniform_int8(seed, N * C * H * W, lo, hi).reshape(N, C, H, W)
    f = synth.uniform_int8(seed + 1, K * C * R * S, lo, hi).reshape(K, C, R, S)
    return x, f


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("alpha", [2.0 ** -9, 1.0 / 3.0])
@pytest.mark.parametrize("kernel", [dict(kernel_variant=1), dict(kernel_variant=2),
                                    dict(kernel_variant=2, halo_loads=1), dict(kernel_variant=2, halo_loads=2),
                                    dict(kernel_variant=3), dict(kernel_variant=3, block_n=64),
                                    dict(kernel_variant=3, block_n=256, halo_loads=1),
                                    dict(kernel_variant=2, halo_loads=3), dict(kernel_variant=3, halo_loads=3),
                                    dict(kernel_variant=3, block_n=64, halo_loads=3)],
                         ids=["gather", "halo", "halo-staged", "halo-direct", "pair", "pair-64", "pair-256-staged",
                              "halo-tma", "pair-tma", "pair-64-tma"])
def test_small_shapes_exact(shape, alpha, kernel):
    x, f = _data(shape, 1000 + sum(shape))
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, alpha)
    y, acc = gpu_util.gpu_run(shape, x, f, alpha, **kernel)
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("opts", [
    dict(num_ctas=1), dict(num_ctas=3), dict(max_chunk_slices=1), dict(max_chunk_slices=5),
    dict(block_n=32), dict(block_n=64), dict(block_n=128), dict(block_n=256, num_ctas=2),
    dict(kernel_variant=1, num_ctas=1), dict(kernel_variant=1, max_chunk_slices=5),
    dict(kernel_variant=1, block_n=64), dict(kernel_variant=2, block_n=256, max_chunk_slices=7),
    dict(kernel_variant=2, block_n=32, num_ctas=5), dict(kernel_variant=2, block_n=256, halo_loads=2),
    dict(kernel_variant=2, block_n=128, halo_loads=1, num_ctas=7),
    # 256 wide with the staging ring: one fp16 halo stage beside two staging slots
    dict(kernel_variant=2, block_n=256, halo_loads=1), dict(kernel_variant=2, block_n=256, halo_loads=1, num_ctas=5),
    dict(kernel_variant=3, num_ctas=2), dict(kernel_variant=3, num_ctas=6, max_chunk_slices=3),
    dict(kernel_variant=3, block_n=128, max_chunk_slices=1), dict(kernel_variant=3, block_n=256, num_ctas=4),
], ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_plan_options_exact(opts):
    shape = (2, 128, 23, 23, 256, 3, 3, 1, 1, 2, 2, 1, 1)
    x, f = _data(shape, 77)
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -10)
    y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -10, **opts)
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    assert np.array_equal(y, y_ref)


EXTREME_SHAPE = (1, 1024, 8, 8, 256, 3, 3, 1, 1, 1, 1, 1, 1)   # 288 K-slices: chunks of 27 to 32 slices


def _extreme_data(shape):
    """Every product near 2^14 (x = f = -128, with -127 sprinkled in to make
    odd sums), and one output channel of large negative sums: an interior
    chunk of c K-slices sums to nearly c * 32 * 2^14, just below 2^24 for
    c = 32."""
    N, C, H, W, K, R, S = shape[:7]
    x = np.full((N, C, H, W), -128, np.int8)
    f = np.full((K, C, R, S), -128, np.int8)
    rng = np.random.default_rng(9)
    x.reshape(-1)[rng.choice(x.size, 97, replace=False)] = -127
    f.reshape(-1)[rng.choice(f.size, 501, replace=False)] = -127
    f[3] = 127
    return x, f


@pytest.mark.parametrize("kw", [dict(kernel_variant=6), dict(kernel_variant=6, max_chunk_slices=6)],
                         ids=["stacked", "stacked-short-chunks"])
def test_extreme_magnitudes_exact_stacked(kw):
    """The stacked-tap kernel (64 output channels, two taps per MMA): chunks
    of 16 filter rows of a 3x3 filter put 16 x 2 taps x 32 channels = 1024
    products near 2^14 into a column, sums at 2^24, and the int32 running
    sums of both column blocks must add up exactly."""
    shape = (1, 1024, 8, 8, 64, 3, 3, 1, 1, 1, 1, 1, 1)
    x, f = _extreme_data(shape)
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -20)
    assert np.abs(acc_ref).max() > 2 ** 27
    y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -20, **kw)
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("kw", [dict(kernel_variant=1), dict(kernel_variant=2), dict(kernel_variant=2, block_n=64),
                                dict(kernel_variant=3), dict(kernel_variant=3, block_n=256),
                                dict(kernel_variant=4), dict(kernel_variant=4, tile_px=256),
                                dict(kernel_variant=5), dict(kernel_variant=5, tile_px=128),
                                dict(kernel_variant=4, filter_run=3, max_chunk_slices=30),
                                dict(kernel_variant=2, halo_loads=3), dict(kernel_variant=3, halo_loads=3),
                                dict(kernel_variant=4, halo_loads=3), dict(kernel_variant=5, halo_loads=3)],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_extreme_magnitudes_exact(kw):
    """Products near 2^14 and odd chunk sums just below 2^24 on every kernel
    form (per-tap gather, halo, halo on CTA pairs, transposed tiles on single
    CTAs and on pairs): the fp32 tensor-core accumulation must stay exact
    chunk by chunk, and the int32 running sums (tensor memory in the gather
    kernel, epilogue registers in the others) must add the chunks exactly."""
    shape = EXTREME_SHAPE
    x, f = _extreme_data(shape)
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -20)
    assert np.abs(acc_ref).max() > 2 ** 27
    y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -20, **kw)
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("variant", [1, 2, 3, 4, 5], ids=["gather", "halo", "halo-pair", "transposed",
                                                          "transposed-pair"])
def test_saturation_and_ties(variant):
    """Alphas that saturate everything (1e30), flip signs (-1), zero every
    output (0), or leave many exact .5 ties (powers of two): every int8 output
    equals the oracle's, on every kernel form."""
    shape = (1, 64, 12, 12, 256, 3, 3, 1, 1, 1, 1, 1, 1)
    x, f = _data(shape, 5)
    for alpha in (1.0, 2.0 ** -9, 2.0 ** -14, 1e30, -1.0, 0.0, -2.0 ** -11):
        y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, alpha)
        y, _ = gpu_util.gpu_run(shape, x, f, alpha, want_acc=False, kernel_variant=variant)
        assert np.array_equal(y, y_ref), alpha


def test_deterministic_repeat():
    import torch
    import int8_implicit_gemm_gb300 as ext
    shape = (4, 256, 14, 14, 256, 3, 3, 1, 1, 1, 1, 1, 1)
    x, f = _data(shape, 21)
    xp, fp = gpu_util.packed_inputs(x, f)
    xd, fd = torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda()
    plan = ext.Plan(shape)
    outs = []
    for _ in range(3):
        y = torch.empty(4 * 256 * 14 * 14, dtype=torch.int8, device="cuda")
        plan.run(xd, fd, y, 2.0 ** -12)
        outs.append(y.cpu().numpy())
    assert plan.status() == 0
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


_FULL_ORACLE = {}


def _full_oracle(wl):
    """The oracle's int32 accumulators and int8 outputs of a whole workload,
    packed NCxHWx<32>; computed once per workload (the tests below take the
    workloads one after another, so only the current one is kept)."""
    if wl.name not in _FULL_ORACLE:
        _FULL_ORACLE.clear()
        x = wl.activations_nchw()
        f = wl.filters_kcrs()
        y, acc = oracle.Oracle().conv2d_fprop(x, f, wl.shape_tuple(), wl.alpha)
        acc32 = acc.astype(np.int32)
        del acc
        _FULL_ORACLE[wl.name] = (oracle.nchw_to_ncxhwx32(y), oracle.nchw_to_ncxhwx32(acc32), x, f)
    return _FULL_ORACLE[wl.name]


@pytest.mark.parametrize("kw", [{}, dict(kernel_variant=2, halo_loads=1), dict(kernel_variant=2, halo_loads=2),
                                dict(kernel_variant=3), dict(kernel_variant=4), dict(kernel_variant=5),
                                dict(kernel_variant=6), dict(kernel_variant=2, halo_loads=3),
                                dict(kernel_variant=3, halo_loads=3), dict(kernel_variant=4, halo_loads=3),
                                dict(kernel_variant=5, halo_loads=3), dict(fused_filter=3),
                                dict(kernel_variant=2, fused_filter=2)],
                         ids=["auto", "staged", "direct", "pair", "transposed", "transposed-pair", "stacked",
                              "halo-tma", "pair-tma", "transposed-tma", "transposed-pair-tma", "filter-conversion-kernel",
                              "single-filter-in-kernel"])
@pytest.mark.parametrize("wl", synth.WORKLOADS, ids=lambda w: w.name)
def test_full_size_workloads(wl, kw):
    """The five workloads at full size, in the launch configuration the
    benchmark times (auto), with each halo load form forced and on CTA pairs:
    every int32 accumulator and every int8 output against the oracle's."""
    import int8_implicit_gemm_gb300 as ext
    shape = wl.shape_tuple()
    if kw:
        try:
            ext.Plan(shape, **kw).destroy()
        except ext.I8ConvError as e:
            if e.status == ext.I8C_ERR_UNSUPPORTED:
                pytest.skip("this kernel form does not fit")
            raise
    y_ref, acc_ref, x, f = _full_oracle(wl)
    y, acc = gpu_util.gpu_run(shape, x, f, wl.alpha, **kw)
    assert np.array_equal(acc, acc_ref)
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("kw", [dict(num_ctas=10), dict(num_ctas=16), dict(kernel_variant=3, num_ctas=6),
                                dict(kernel_variant=2, block_n=32, num_ctas=9, max_chunk_slices=4)],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_split_tail_exact(kw):
    """Tiles of a partial last wave split along the channel blocks: the units'
    int32 partial sums, combined by the unit that finishes last, give the
    oracle's results exactly (and the same as without splitting)."""
    import int8_implicit_gemm_gb300 as ext
    shape = (2, 512, 7, 6, 64, 3, 3, 1, 1, 1, 1, 1, 1)   # 16 channel blocks, 2 patches
    plan = ext.Plan(shape, tail_split=2, **kw)
    assert plan.info["tail_split"] > 1, plan.info
    plan.destroy()
    x, f = _data(shape, 4242)
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -12)
    for ts in (2, 1, 2):   # split, unsplit, split again (counters reset between launches)
        y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -12, tail_split=ts, **kw)
        assert np.array_equal(acc, acc_ref.astype(np.int32)), ts
        assert np.array_equal(y, y_ref), ts


@pytest.mark.parametrize("kw", [dict(block_n=256, num_ctas=9), dict(block_n=128, num_ctas=20), dict(block_n=256, num_ctas=8)],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_halved_tail_exact(kw):
    """Tiles of a partial last wave halved along the output channels (two
    units with N = BN/2 MMAs and disjoint outputs) give the oracle's results."""
    import int8_implicit_gemm_gb300 as ext
    shape = (2, 64, 13, 11, 256, 3, 3, 1, 1, 1, 1, 1, 1)
    plan = ext.Plan(shape, tail_split=3, **kw)
    assert plan.info["tail_halves"] == 2, plan.info
    plan.destroy()
    x, f = _data(shape, 5151)
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -11)
    y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -11, tail_split=3, **kw)
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("shape", [s for s in SMALL if s[9] == 1 and s[10] == 1], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("kw", [dict(kernel_variant=2), dict(kernel_variant=3), dict(kernel_variant=2, halo_loads=1)],
                         ids=["single", "pair", "staged"])
def test_flat_tiles_exact(shape, kw):
    """Tiles of 128 consecutive pixels of the padded row-major output (stride
    1): every real output pixel exact, the discarded ones never stored."""
    x, f = _data(shape, 777 + sum(shape))
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -9)
    y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -9, tile_shape=2, **kw)
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    assert np.array_equal(y, y_ref)


TRANSPOSED_EXTRA = [
    (2, 64, 20, 20, 128, 3, 3, 1, 1, 1, 1, 1, 1),     # 400 pixels per image over several tiles
    (1, 96, 9, 33, 224, 3, 3, 1, 1, 1, 1, 1, 1),      # K = 224: the second channel tile half empty
]


@pytest.mark.parametrize("shape", [s for s in SMALL if s[9] == 1 and s[10] == 1] + TRANSPOSED_EXTRA,
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("kw", [dict(), dict(tile_px=16), dict(tile_px=176), dict(tile_px=256),
                                dict(tile_px=64, filter_run=3), dict(tile_px=128, filter_run=1, max_chunk_slices=5),
                                dict(num_ctas=3, tile_px=96), dict(halo_loads=1), dict(tile_px=240, halo_loads=1),
                                dict(halo_loads=3), dict(tile_px=176, halo_loads=3), dict(tile_px=64, halo_loads=3)],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()) or "auto")
@pytest.mark.parametrize("variant", [4, 5], ids=["single", "pair"])
def test_transposed_tiles_exact(shape, kw, variant):
    """Transposed tiles (128 output channels per CTA on the MMA's M, tile_px
    output pixels on N, stride 1; on CTA pairs M = 256 and each CTA builds
    the halo of half the pixels): every output exact for every tile width,
    filter stage length, chunk length, grid size and load form."""
    import int8_implicit_gemm_gb300 as ext
    if variant == 5 and "num_ctas" in kw:
        kw = dict(kw, num_ctas=2 * kw["num_ctas"])
    try:
        ext.Plan(shape, kernel_variant=variant, **kw).destroy()
    except ext.I8ConvError as e:
        if e.status == ext.I8C_ERR_UNSUPPORTED and "filter_run" in kw:
            pytest.skip("the forced filter stage length does not divide R*S")
        raise
    x, f = _data(shape, 2024 + sum(shape))
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -9)
    y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -9, kernel_variant=variant, **kw)
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("variant", [4, 5])
def test_transposed_tiles_rejects_strides(variant):
    import int8_implicit_gemm_gb300 as ext
    with pytest.raises(ext.I8ConvError) as ei:
        ext.Plan((2, 128, 23, 23, 256, 3, 3, 1, 1, 2, 2, 1, 1), kernel_variant=variant)
    assert ei.value.status == ext.I8C_ERR_UNSUPPORTED


def _channel_params(K, seed):
    """Per-channel scales (powers of two and arbitrary values) and biases
    (quarter steps that make .5 ties, and arbitrary values)."""
    rng = np.random.default_rng(seed)
    scale = np.where(rng.random(K) < 0.5, 2.0 ** rng.integers(-13, -6, K),
                     rng.uniform(1e-4, 4e-3, K)).astype(np.float32)
    bias = np.where(rng.random(K) < 0.5, rng.integers(-80, 81, K) / 4.0,
                    rng.uniform(-40.0, 40.0, K)).astype(np.float32)
    return scale, bias


@pytest.mark.parametrize("variant", [1, 2, 3, 4, 5], ids=["gather", "halo", "halo-pair", "transposed",
                                                          "transposed-pair"])
@pytest.mark.parametrize("ep", [dict(scale=True), dict(bias=True), dict(scale=True, bias=True, relu=True),
                                dict(relu=True)], ids=["scale", "bias", "scale-bias-relu", "relu"])
def test_channel_epilogue_exact(variant, ep):
    """The per-output-channel epilogue (scale, bias, ReLU before the clamp)
    on every kernel form: every int8 output equals the oracle's."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    shape = (2, 64, 13, 11, 256, 3, 3, 1, 1, 1, 1, 1, 1)
    N, C, H, W, K = shape[:5]
    x, f = _data(shape, 4321)
    orc = oracle.Oracle()
    acc = orc.conv_acc(x, f, shape)
    scale, bias = _channel_params(K, 99)
    alpha = 2.0 ** -10
    y_ref = orc.requantize_channels(acc, alpha, scale if ep.get("scale") else None,
                                    bias if ep.get("bias") else None, ep.get("relu", False))
    xp, fp = gpu_util.packed_inputs(x, f)
    xd, fd = torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda()
    plan = ext.Plan(shape, kernel_variant=variant)
    P, Q = plan.info["P"], plan.info["Q"]
    y = torch.full((N, K // 32, P, Q, 32), 77, dtype=torch.int8, device="cuda")
    sd = torch.from_numpy(scale).cuda() if ep.get("scale") else None
    bd = torch.from_numpy(bias).cuda() if ep.get("bias") else None
    plan.run(xd, fd, y, alpha, alpha_k=sd, bias=bd, relu=ep.get("relu", False))
    torch.cuda.synchronize()
    assert plan.status() == 0
    plan.destroy()
    assert np.array_equal(y.cpu().numpy(), oracle.nchw_to_ncxhwx32(y_ref))


def test_channel_epilogue_full_size_bench_workload():
    """The benchmark workload at full size with per-channel scales, biases and
    ReLU, in its auto launch configuration: the int32 accumulators against
    the oracle at sampled points, and y == the oracle's per-channel epilogue
    of those accumulators at every output element."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    wl = synth.WORKLOADS_BY_NAME["n8c256h56k256r3s1"]
    shape = wl.shape_tuple()
    x = wl.activations_nchw()
    f = wl.filters_kcrs()
    xp, fp = gpu_util.packed_inputs(x, f)
    xd, fd = torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda()
    plan = ext.Plan(shape)
    P, Q = plan.info["P"], plan.info["Q"]
    N, K = wl.N, wl.K
    scale, bias = _channel_params(K, 7)
    y = torch.empty((N, K // 32, P, Q, 32), dtype=torch.int8, device="cuda")
    acc = torch.empty((N, K // 32, P, Q, 32), dtype=torch.int32, device="cuda")
    plan.run(xd, fd, y, wl.alpha, alpha_k=torch.from_numpy(scale).cuda(), bias=torch.from_numpy(bias).cuda(),
             relu=True)
    plan.run_acc(xd, fd, acc)
    torch.cuda.synchronize()
    assert plan.status() == 0
    plan.destroy()
    orc = oracle.Oracle()
    acc_np = acc.cpu().numpy()
    pts = gpu_util.sample_points(shape, P, Q, 2000, seed=5)
    idx = gpu_util.packed_index(shape, P, Q, pts)
    assert np.array_equal(acc_np.reshape(-1)[idx].astype(np.int64), orc.conv_acc_points(x, f, shape, pts))
    acc_nkpq = oracle.ncxhwx32_to_nchw(acc_np, N, K, P, Q).astype(np.int64)
    y_ref = orc.requantize_channels(acc_nkpq, wl.alpha, scale, bias, relu=True)
    assert np.array_equal(y.cpu().numpy(), oracle.nchw_to_ncxhwx32(y_ref))


@pytest.mark.parametrize("shape,opts", [
    ((2, 32, 40, 40, 64, 5, 9, 2, 4, 1, 1, 2, 3), dict(kernel_variant=3, block_n=64, num_ctas=4)),
    ((2, 32, 40, 40, 32, 5, 9, 2, 4, 1, 1, 2, 3), dict(kernel_variant=2, block_n=32, num_ctas=3)),
    ((3, 64, 20, 20, 64, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=2, block_n=64, num_ctas=2)),
    ((2, 96, 17, 17, 32, 3, 3, 1, 1, 2, 2, 1, 1), dict(kernel_variant=2, num_ctas=2)),
    ((1, 32, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1), dict(num_ctas=1)),
    ((2, 64, 20, 20, 32, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=2, block_n=64, num_ctas=2)),
    ((2, 32, 24, 24, 32, 5, 9, 2, 4, 1, 1, 2, 3), dict(kernel_variant=3, block_n=64, num_ctas=2)),
    ((2, 64, 24, 40, 32, 3, 3, 1, 1, 1, 1, 1, 1), dict(tile_shape=3, num_ctas=2)),
], ids=["dilated-pair", "dilated-single", "3x3-two-blocks", "stride2-three-blocks", "16x16",
        "rows-past-K", "pair-rows-past-K", "wide-patches"])
@pytest.mark.parametrize("fused", [3, 2, 0], ids=["tma", "in-kernel", "auto"])
def test_resident_filter_exact(shape, opts, fused):
    """One output-channel tile and whole-tile units: the filter stages are
    loaded once per CTA and reused by every later tile (few CTAs, so each runs
    many tiles), either by TMA from the fp16 copy the conversion kernel wrote
    (fused_filter = 3) or written by the kernel's own threads straight from
    the int8 filter before the warp roles split (fused_filter = 2, the auto
    choice for a resident filter; the tile's rows past K are zeros);
    bit-exact against the oracle."""
    import int8_implicit_gemm_gb300 as ext
    opts = dict(opts, fused_filter=fused)
    opts.setdefault("tile_shape", 1)  # 16x8 tiles unless the case asks for 16x16 patches: many units per CTA
    try:
        plan = ext.Plan(shape, **opts)
    except ext.I8ConvError as e:
        if e.status == ext.I8C_ERR_UNSUPPORTED and shape[4] < opts.get("block_n", 0):
            pytest.skip("block_n wider than K is not planned")
        raise
    assert plan.info["kernels_per_run"] == (2 if fused == 3 else 1)
    assert plan.info["filter_resident"] == 1
    assert plan.info["work_units"] > plan.info["num_ctas"] // (2 if plan.info["kernel_variant"] == 3 else 1)
    plan.destroy()
    x, f = _data(shape, 4242 + sum(shape))
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -10)
    y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -10, **opts)
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    assert np.array_equal(y, y_ref)


STACKED_SHAPES = [
    # N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw        (K = 64, stride 1)
    (2, 32, 40, 300, 64, 5, 9, 2, 4, 1, 1, 2, 3),       # the dilated 5x9 layer's geometry, ragged row tiles
    (2, 32, 17, 130, 64, 3, 3, 1, 1, 1, 1, 1, 1),       # odd S, shift 1, two tiles per row
    (1, 64, 9, 250, 64, 2, 2, 0, 1, 1, 1, 1, 2),        # even S (no single tap), two channel blocks
    (3, 96, 6, 40, 64, 3, 5, 1, 2, 1, 1, 1, 1),         # three channel blocks, one tile per row
    (1, 32, 12, 128, 64, 1, 7, 0, 3, 1, 1, 1, 8),       # R = 1, the largest shift (8)
    (2, 32, 5, 5, 64, 3, 3, 1, 1, 1, 1, 1, 1),          # tiny image: most of the tile outside the row
    (1, 32, 6, 200, 64, 4, 16, 1, 7, 1, 1, 1, 1),       # S = 16: eight tap pairs per row
    (1, 160, 7, 64, 64, 3, 3, 1, 1, 1, 1, 2, 2),        # five channel blocks: several chunks of rows
]


@pytest.mark.parametrize("shape", STACKED_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("kw", [dict(), dict(num_ctas=2), dict(num_ctas=6, max_chunk_slices=4)],
                         ids=["default", "one-pair", "three-pairs-short-chunks"])
def test_stacked_taps_exact(shape, kw):
    """The stacked-tap kernel (two filter taps per N = 128 MMA, the second
    tap's column block shifted by dw pixels in the epilogue, row tiles of
    128 - dw valid outputs, CTA pairs): every int32 accumulator and int8 output
    exact, for odd and even filter widths, shifts 1 to 8, several channel
    blocks and chunks, and few CTAs running many tiles on a resident filter."""
    x, f = _data(shape, 3131 + sum(shape))
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -10)
    y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -10, kernel_variant=6, **kw)
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("ep", [dict(scale=True, bias=True, relu=True), dict(bias=True)], ids=["scale-bias-relu", "bias"])
def test_stacked_taps_channel_epilogue(ep):
    import torch
    import int8_implicit_gemm_gb300 as ext
    shape = (2, 32, 20, 150, 64, 5, 9, 2, 4, 1, 1, 2, 3)
    N, C, H, W, K = shape[:5]
    x, f = _data(shape, 4343)
    orc = oracle.Oracle()
    acc = orc.conv_acc(x, f, shape)
    scale, bias = _channel_params(K, 98)
    alpha = 2.0 ** -10
    y_ref = orc.requantize_channels(acc, alpha, scale if ep.get("scale") else None,
                                    bias if ep.get("bias") else None, ep.get("relu", False))
    xp, fp = gpu_util.packed_inputs(x, f)
    xd, fd = torch.from_numpy(xp).cuda(), torch.from_numpy(fp).cuda()
    plan = ext.Plan(shape, kernel_variant=6)
    P, Q = plan.info["P"], plan.info["Q"]
    y = torch.full((N, K // 32, P, Q, 32), 77, dtype=torch.int8, device="cuda")
    sd = torch.from_numpy(scale).cuda() if ep.get("scale") else None
    bd = torch.from_numpy(bias).cuda() if ep.get("bias") else None
    plan.run(xd, fd, y, alpha, alpha_k=sd, bias=bd, relu=ep.get("relu", False))
    torch.cuda.synchronize()
    assert plan.status() == 0
    plan.destroy()
    assert np.array_equal(y.cpu().numpy(), oracle.nchw_to_ncxhwx32(y_ref))


def test_stacked_taps_rejects_unsuited_shapes():
    import int8_implicit_gemm_gb300 as ext
    for shape in [(1, 32, 16, 16, 128, 3, 3, 1, 1, 1, 1, 1, 1),     # K != 64
                  (1, 32, 16, 16, 64, 3, 3, 1, 1, 2, 2, 1, 1),      # stride 2
                  (1, 32, 16, 16, 64, 3, 1, 1, 0, 1, 1, 1, 1),      # S = 1: no tap pairs
                  (1, 32, 40, 40, 64, 3, 3, 1, 9, 1, 1, 1, 9)]:     # shift 9 > 8
        with pytest.raises(ext.I8ConvError) as ei:
            ext.Plan(shape, kernel_variant=6)
        assert ei.value.status == ext.I8C_ERR_UNSUPPORTED, shape


@pytest.mark.parametrize("shape,kw", [
    ((2, 64, 13, 11, 96, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=1)),
    ((2, 64, 13, 11, 96, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=2)),
    ((2, 64, 13, 11, 128, 3, 3, 1, 1, 2, 2, 1, 1), dict(kernel_variant=3)),
    ((2, 64, 13, 11, 128, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=4)),
    ((2, 64, 13, 11, 256, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=5)),
    ((2, 64, 12, 40, 64, 3, 5, 1, 2, 1, 1, 1, 1), dict(kernel_variant=6)),
    ((2, 96, 13, 11, 128, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=2, fused_filter=1)),
    ((2, 32, 24, 24, 64, 5, 9, 2, 4, 1, 1, 2, 3), dict(kernel_variant=3, fused_filter=2)),
    ((2, 32, 24, 24, 64, 5, 9, 2, 4, 1, 1, 2, 3), dict(kernel_variant=3, fused_filter=3)),
], ids=["gather", "halo", "halo-pair-s2", "transposed", "transposed-pair", "stacked", "grid-barrier-filter",
        "resident-in-kernel", "resident-tma"])
def test_prepacked_filter_exact(shape, kw):
    """Weight prepacking: set_filter converts the filter once, run_prepacked
    runs the convolution alone; outputs bit-exact against the oracle on two
    different activations, unchanged after the caller overwrites its filter
    buffer, with the per-channel epilogue too; an ordinary run with another
    filter withdraws the prepacked copy."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    N, C, H, W, K = shape[:5]
    x1, f = _data(shape, 9100 + sum(shape))
    x2, _ = _data(shape, 9200 + sum(shape))
    orc = oracle.Oracle()
    try:
        plan = ext.Plan(shape, **kw)
    except ext.I8ConvError as e:
        if e.status == ext.I8C_ERR_UNSUPPORTED:
            pytest.skip("plan form not available for this shape")
        raise
    P, Q = plan.info["P"], plan.info["Q"]
    xp1, fp = gpu_util.packed_inputs(x1, f)
    xp2, _ = gpu_util.packed_inputs(x2, f)
    fd = torch.from_numpy(fp).cuda()
    xd1, xd2 = torch.from_numpy(xp1).cuda(), torch.from_numpy(xp2).cuda()
    y = torch.full((N, K // 32, P, Q, 32), 55, dtype=torch.int8, device="cuda")
    with pytest.raises(ext.I8ConvError):
        plan.run_prepacked(xd1, y, 2.0 ** -10)   # no filter set yet
    plan.set_filter(fd)
    fd.zero_()                                    # the plan keeps its own copy
    for xd, xn in ((xd1, x1), (xd2, x2)):
        plan.run_prepacked(xd, y, 2.0 ** -10)
        torch.cuda.synchronize()
        y_ref, _ = gpu_util.oracle_packed(shape, xn, f, 2.0 ** -10)
        assert np.array_equal(y.cpu().numpy(), y_ref)
    rng = np.random.default_rng(11)
    scale = rng.uniform(2.0 ** -12, 2.0 ** -8, K).astype(np.float32)
    bias = rng.uniform(-40, 40, K).astype(np.float32)
    plan.run_prepacked(xd2, y, 1.0, alpha_k=torch.from_numpy(scale).cuda(), bias=torch.from_numpy(bias).cuda(),
                       relu=True)
    torch.cuda.synchronize()
    acc = orc.conv2d_fprop(x2, f, shape, 1.0)[1].astype(np.int64)
    assert np.array_equal(y.cpu().numpy(), oracle.nchw_to_ncxhwx32(orc.requantize_channels(acc, 1.0, scale, bias,
                                                                                            relu=True)))
    plan.run(xd1, fd, y, 2.0 ** -10)              # an ordinary run with the (zeroed) filter
    torch.cuda.synchronize()
    assert not y.cpu().numpy().any()
    with pytest.raises(ext.I8ConvError):
        plan.run_prepacked(xd1, y, 2.0 ** -10)
    assert plan.status() == 0
    plan.destroy()


@pytest.mark.parametrize("kw", [dict(kernel_variant=2), dict(kernel_variant=3), dict(kernel_variant=4),
                                dict(kernel_variant=6), dict(kernel_variant=2, fused_filter=2)],
                         ids=["halo", "halo-pair", "transposed", "stacked", "resident-in-kernel"])
@pytest.mark.parametrize("prepacked", [False, True], ids=["runs", "prepacked"])
def test_chained_runs_ping_pong(kw, prepacked):
    """Each run reads the previous run's output and writes the buffer the run
    before it read (two buffers, six runs back to back on one stream): the
    dependent launches must order every activation read after the previous
    kernel's writes and every output write after its reads.  Bit-exact
    against the oracle applied six times."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    shape = (2, 64, 16, 16, 64, 3, 3, 1, 1, 1, 1, 1, 1)
    x, f = _data(shape, 4711)
    try:
        plan = ext.Plan(shape, **kw)
    except ext.I8ConvError as e:
        if e.status == ext.I8C_ERR_UNSUPPORTED:
            pytest.skip("plan form not available for this shape")
        raise
    xp, fp = gpu_util.packed_inputs(x, f)
    fd = torch.from_numpy(fp).cuda()
    bufs = [torch.from_numpy(xp).cuda(), torch.empty_like(torch.from_numpy(xp)).cuda()]
    alpha = 2.0 ** -11  # keeps six generations spread out (mean |y| about 19, none saturated)
    if prepacked:
        plan.set_filter(fd)
    for i in range(6):
        src, dst = bufs[i % 2], bufs[(i + 1) % 2]
        if prepacked:
            plan.run_prepacked(src, dst, alpha)
        else:
            plan.run(src, fd, dst, alpha)
    torch.cuda.synchronize()
    assert plan.status() == 0
    orc = oracle.Oracle()
    cur = x
    for _ in range(6):
        cur = orc.conv2d_fprop(cur, f, shape, alpha)[0]
    assert np.array_equal(bufs[0].cpu().numpy(), oracle.nchw_to_ncxhwx32(cur))
    plan.destroy()


@pytest.mark.parametrize("kw", [dict(kernel_variant=4), dict(kernel_variant=3), dict(kernel_variant=6),
                                dict(kernel_variant=3, fused_filter=2), dict(kernel_variant=2, fused_filter=1)],
                         ids=["transposed", "halo-pair", "stacked", "resident-in-kernel", "grid-barrier-filter"])
def test_prepacked_filter_switch_on_one_stream(kw):
    """set_filter with a second filter right after prepacked runs with the
    first, then a prepacked run at once on the same stream: the conversion (or
    copy) of the new filter is the work just before that run's kernel, which
    must wait for it before reading the filter; alternating three times, each
    run bit-exact against the oracle with its own filter."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    shape = (2, 64, 12, 40, 64, 3, 5, 1, 2, 1, 1, 1, 1)
    N, C, H, W, K = shape[:5]
    x, f1 = _data(shape, 7100)
    _, f2 = _data(shape, 7200)
    try:
        plan = ext.Plan(shape, **kw)
    except ext.I8ConvError as e:
        if e.status == ext.I8C_ERR_UNSUPPORTED:
            pytest.skip("plan form not available for this shape")
        raise
    P, Q = plan.info["P"], plan.info["Q"]
    xp, fp1 = gpu_util.packed_inputs(x, f1)
    _, fp2 = gpu_util.packed_inputs(x, f2)
    xd = torch.from_numpy(xp).cuda()
    fds = [torch.from_numpy(fp1).cuda(), torch.from_numpy(fp2).cuda()]
    refs = [gpu_util.oracle_packed(shape, x, ff, 2.0 ** -10)[0] for ff in (f1, f2)]
    ys = [torch.full((N, K // 32, P, Q, 32), 33, dtype=torch.int8, device="cuda") for _ in range(6)]
    s = torch.cuda.current_stream()
    for i in range(6):
        plan.set_filter(fds[i % 2], s)
        plan.run_prepacked(xd, ys[i], 2.0 ** -10, s)
        plan.run_prepacked(xd, ys[i], 2.0 ** -10, s)   # a second run: no wait for the filter
    torch.cuda.synchronize()
    assert plan.status() == 0
    for i in range(6):
        assert np.array_equal(ys[i].cpu().numpy(), refs[i % 2]), i
    plan.destroy()


WIDE_SHAPES = [
    (2, 32, 24, 40, 64, 5, 9, 2, 4, 1, 1, 2, 3),    # the dilated 5x9 layer's geometry, small
    (2, 64, 20, 37, 64, 3, 3, 1, 1, 1, 1, 1, 1),    # ragged last patch column
    (1, 32, 33, 45, 32, 3, 3, 1, 1, 2, 2, 1, 1),    # stride 2
    (2, 96, 35, 37, 256, 3, 3, 1, 1, 2, 2, 1, 1),   # stride 2, three channel blocks, two 128-wide channel tiles
    (1, 64, 21, 30, 160, 3, 3, 1, 1, 1, 1, 1, 1),   # K = 160: a ragged 128-wide channel tile
]


@pytest.mark.parametrize("shape", WIDE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("kw", [dict(tile_shape=3), dict(tile_shape=3, kernel_variant=3),
                                dict(tile_shape=3, kernel_variant=3, num_ctas=4),
                                dict(tile_shape=3, kernel_variant=3, halo_loads=1),
                                dict(tile_shape=3, kernel_variant=2, block_n=128),
                                dict(tile_shape=3, kernel_variant=3, block_n=128, num_ctas=6)],
                         ids=["auto", "pair", "pair-4-ctas", "pair-staged", "single-128", "pair-128"])
def test_wide_patches_exact(shape, kw):
    """16x16 patches (two 16x8 sub-tiles on one halo, two MMAs per tap and K
    half into an accumulator pair): every int32 accumulator and int8 output
    bit-exact against the oracle, ragged patch columns included."""
    import int8_implicit_gemm_gb300 as ext
    try:
        plan = ext.Plan(shape, **kw)
    except ext.I8ConvError as e:
        if e.status == ext.I8C_ERR_UNSUPPORTED:
            pytest.skip("16x16 patches not available for this plan form")
        raise
    assert plan.layout()["subtiles"] == 2
    plan.destroy()
    x, f = _data(shape, 9900 + sum(shape))
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -10)
    y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -10, **kw)
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    assert np.array_equal(y, y_ref)


def _random_small_shapes(seed, count):
    """Seeded small convolutions across the planner's ranges (strides and
    dilations 1-4, filters up to 7 taps a side, paddings up to the filter's
    reach, ragged images, K a multiple of 32), sized for the oracle."""
    import random
    rng = random.Random(seed)
    out = []
    while len(out) < count:
        R, S = rng.randint(1, 7), rng.randint(1, 7)
        sh, sw = rng.choice([1, 1, 2, 3, 4]), rng.choice([1, 1, 2, 3, 4])
        if rng.random() < 0.4:  # stride 1 both ways: the transposed and stacked forms too
            sh = sw = 1
        dh, dw = rng.choice([1, 1, 2, 3]), rng.choice([1, 1, 2, 4])
        ph, pw = rng.randint(0, (R - 1) * dh), rng.randint(0, (S - 1) * dw)
        H, W = rng.randint(3, 30), rng.randint(3, 40)
        N, C, K = rng.randint(1, 3), 32 * rng.randint(1, 3), 32 * rng.randint(1, 4)
        P = (H + 2 * ph - dh * (R - 1) - 1) // sh + 1
        Q = (W + 2 * pw - dw * (S - 1) - 1) // sw + 1
        if P >= 1 and Q >= 1:
            out.append((N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw))
    return out


RANDOM_FORMS = [{}, dict(kernel_variant=1), dict(kernel_variant=2), dict(kernel_variant=3),
                dict(kernel_variant=4), dict(kernel_variant=5), dict(kernel_variant=6),
                dict(kernel_variant=2, halo_loads=3), dict(tile_shape=3), dict(kernel_variant=2, halo_loads=1)]


@pytest.mark.parametrize("shape", _random_small_shapes(2024, 24), ids=lambda s: "x".join(map(str, s)))
def test_random_shapes_exact(shape):
    """Seeded random small shapes on every kernel form the planner accepts for
    them (auto, per-tap gather, halo, halo pairs, transposed tiles on single
    CTAs and pairs, stacked taps, TMA-fed halos, 16x16 patches, staged
    halos): int32 accumulators and int8 outputs bit-exact against the oracle;
    forms the planner refuses are skipped."""
    import int8_implicit_gemm_gb300 as ext
    x, f = _data(shape, 31 + sum(shape))
    y_ref, acc_ref = gpu_util.oracle_packed(shape, x, f, 2.0 ** -10)
    ran = 0
    for kw in RANDOM_FORMS:
        try:
            ext.Plan(shape, **kw).destroy()
        except ext.I8ConvError as e:
            if e.status == ext.I8C_ERR_UNSUPPORTED:
                continue
            raise
        y, acc = gpu_util.gpu_run(shape, x, f, 2.0 ** -10, **kw)
        assert np.array_equal(acc, acc_ref.astype(np.int32)), kw
        assert np.array_equal(y, y_ref), kw
        ran += 1
    assert ran >= 2
