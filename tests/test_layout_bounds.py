"""Host-side bounds check of the kernels' shared- and tensor-memory layouts.

compute-sanitizer is not available for these kernels, so this CPU test stands
in for its out-of-bounds check: for every plan form the parity tests run, and
for the five workloads, it takes the layout the planner gives the kernel
(i8c_plan_layout: the same planner as i8c_plan_create, run on the host with
no GPU) and computes, from the convolution's geometry alone, the furthest
byte that each access can reach:

* the activation operand's matrix descriptors: the shifted halo view of every
  filter tap, over all 8-row core-matrix groups (stride SBO) and both 8-channel
  planes of each 16-channel MMA step (distance LBO), for both MMAs of a K-slice;
* the filter operand's descriptors and the filter TMA box of every stage;
* the halo producers' fp16 stores and the int8 staging ring;
* the transposed-tile epilogue's output staging rows and the barriers;
* the tensor-memory columns of the two accumulator buffers,

and requires each to stay inside its region, the regions to be disjoint and
everything to fit in the shared memory the launch requests.  A planted
off-by-one in a layout must fail the check.
"""
import pytest

import synth
from tests.test_gpu_parity import SMALL, STACKED_SHAPES, TRANSPOSED_EXTRA

KMAX_SMEM = 232448          # opt-in dynamic shared memory per block on sm_103
KMAX_FILTER_STAGES = 16     # filter stages the kernels have barriers for
KHALO_BARRIER_WORDS = 57    # 8-byte barrier and control words the halo and transposed kernels use


def _taps(shape):
    N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw = shape
    return [(r, s) for r in range(R) for s in range(S)]


def check_layout(shape, L):
    """Raise AssertionError if any access of the plan's kernel can leave its region."""
    N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw = shape
    v = L["kernel_variant"]
    assert L["smem_bytes"] <= KMAX_SMEM, "shared memory over the per-block limit"
    tc = L["tmem_cols"]
    assert 32 <= tc <= 512 and tc & (tc - 1) == 0, "tensor-memory allocation must be a power of two in [32, 512]"
    if v == 6:
        return check_stacked_layout(shape, L)
    assert 1 <= L["chunk_slices"] <= 32, "an exact fp32 chunk holds at most 32 K-slices (1024 products)"
    assert L["num_chunks"] * L["chunk_slices"] >= (C // 32) * R * S
    if v == 1:
        BN = L["block_n"]
        st = L["gather_stages"]
        assert L["gather_stage_a"] == 128 * 64 and L["gather_stage_b"] == BN * 64
        assert L["gather_off_a"] + st * L["gather_stage_a"] <= L["gather_off_b"], "A stages overlap B"
        assert L["gather_off_b"] + st * L["gather_stage_b"] <= L["gather_off_staging"], "B stages overlap staging"
        assert L["gather_staging_bytes"] >= 128 * 32
        assert L["gather_off_staging"] + L["gather_staging_slots"] * L["gather_staging_bytes"] <= L["gather_off_bar"]
        assert L["gather_off_bar"] + (3 * st + 5) * 8 + 16 + 1024 <= L["smem_bytes"], "barriers past the allocation"
        run_cols = BN if L["num_chunks"] > 1 else 0
        assert 2 * BN + run_cols <= tc or BN + run_cols <= tc, "accumulators past the tensor-memory allocation"
        return
    CG = L["cta_group"]
    G = L["filter_run"]
    assert L["chunk_slices"] % G == 0, "chunks switch accumulators only between filter stages"
    assert (R * S) % G == 0 or (G <= S and S % G == 0), "a filter stage never spans two channel blocks"
    # filter stages: TMA boxes of G K-slices x rows x 64 bytes, 64-byte swizzled
    rows = 128 if v >= 4 else L["block_n"] // CG
    stage = L["filter_stage_bytes"]
    assert stage == G * rows * 64, "filter stage size"
    assert L["off_filter"] % 1024 == 0, "swizzled filter stages need 1024-byte alignment"
    assert 1 <= L["filter_stages"] <= KMAX_FILTER_STAGES
    filter_end = L["off_filter"] + L["filter_stages"] * stage
    # every B (or transposed A) descriptor: slice t of a stage, both 16-channel halves
    last_slice_end = L["off_filter"] + (L["filter_stages"] - 1) * stage + (G - 1) * rows * 64 + rows * 64
    assert last_slice_end <= filter_end
    # halo stages and the staging ring
    P = (H + 2 * ph - dh * (R - 1) - 1) // sh + 1
    Q = (W + 2 * pw - dw * (S - 1) - 1) // sw + 1
    pos = L["positions"]
    plane = L["plane_bytes"]
    assert L["halo_bytes"] == 4 * plane and plane % 128 == 0, "four 8-channel planes, 128-byte aligned"
    assert plane >= 16 * pos, "a plane holds one 16-byte entry per halo position"
    assert 1 <= L["halo_stages"] <= 3
    assert L["halo_stages"] * L["halo_bytes"] <= L["off_staging"], "halo stages overlap the staging ring"
    if L["staging_slots"] > 0:
        assert L["staging_bytes"] >= 32 * pos
    assert L["off_staging"] + L["staging_slots"] * L["staging_bytes"] <= L["off_filter"], "staging overlaps filter"
    CW = L["halo_cw"]
    if v >= 4 or L["flat_tiles"]:
        # flat tiles: positions m0 + e of the padded row-major image; tap (r, s)
        # starts r*dh*CW + s*dw positions in, and the tile's pixels follow
        assert sh == 1 and sw == 1
        assert CW == W + 2 * pw
        npx = L["tile_px"]
        assert npx % 8 == 0 and npx >= 8
        reach = max(r * dh * CW + s * dw for r, s in _taps(shape)) + npx - 1
        assert pos >= npx + (R - 1) * dh * CW + (S - 1) * dw
    else:
        # 16 x 8 patches (16 x 16 with two sub-tiles side by side): 8-row
        # groups sh halo rows apart, 8 consecutive positions of the tap's
        # column phase within a row, the second sub-tile 8 positions on
        sub = L["subtiles"]
        assert sub in (1, 2)
        last_col = 8 * sub - 1
        assert L["halo_rows"] >= 15 * sh + (R - 1) * dh + 1 and CW >= last_col * sw + (S - 1) * dw + 1
        assert pos == L["halo_rows"] * CW
        ph_off = L["phase_off"]
        assert ph_off[0] == 0 and ph_off[sw] == CW
        reach = 0
        for r, s in _taps(shape):
            f, idx = (s * dw) % sw, (s * dw) // sw
            assert idx + last_col < ph_off[f + 1] - ph_off[f], "a tap's columns run past its column phase"
            reach = max(reach, r * dh * CW + ph_off[f] + idx + 15 * sh * CW + last_col)
    assert reach < pos, f"an operand view reaches halo position {reach} of {pos}"
    # both MMAs of a K-slice: planes 0-1 and 2-3 (start + 2 planes, + LBO = 1 plane)
    assert 3 * plane + 16 * reach + 15 < L["halo_bytes"], "a descriptor reaches past its halo stage"
    end = filter_end
    if v >= 4:
        np_mma = CG * L["tile_px"]
        assert 16 <= np_mma <= 256 and np_mma % 16 == 0, "MMA N"
        assert L["off_out"] >= filter_end, "output staging overlaps the filter stages"
        end = L["off_out"] + 8 * np_mma * 16          # eight epilogue warps, np_mma x 16 bytes each
        assert 2 * np_mma <= tc, "two accumulator buffers of N columns"
        assert L["off_out"] + 8 * np_mma * 16 <= L["off_bar"]
    else:
        assert 2 * L["subtiles"] * L["block_n"] <= tc, "two accumulator buffers of BN columns per sub-tile"
        assert L["tile_px"] in (0, 128)
    assert end <= L["off_bar"], "operands overlap the barriers"
    if L["tma_halo"]:
        check_tma_halo(shape, L, pos)
    assert KHALO_BARRIER_WORDS * 8 <= L["bar_bytes"]
    assert L["off_bar"] + L["bar_bytes"] + 1024 <= L["smem_bytes"], "barriers past the allocation"
    assert P >= 1 and Q >= 1


def check_tma_halo(shape, L, pos):
    """TMA-fed halos: every box (32 bytes x box_w x box_h, at most 256 per
    dimension) fits its int8 slot, the slots sit between the halo stages and
    the filter stages, and every position the converters read lies in the box."""
    N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw = shape
    bw, bh = L["box_w"], L["box_h"]
    assert 1 <= bw <= 256 and 1 <= bh <= 256, "TMA box dimensions"
    assert L["x8_bytes"] >= 32 * bw * bh and L["x8_bytes"] % 1024 == 0
    assert L["x8_slots"] in (1, 2, 3)
    assert L["off_x8"] % 1024 == 0
    assert L["off_x8"] >= L["halo_stages"] * L["halo_bytes"] + L["staging_slots"] * L["staging_bytes"]
    assert L["off_x8"] + L["x8_slots"] * L["x8_bytes"] <= L["off_filter"], "int8 slots overlap the filter"
    CW = L["halo_cw"]
    if L["kernel_variant"] >= 4 or L["flat_tiles"]:
        # a flat run starts anywhere in the box's first padded row
        assert bw == W + 2 * pw == CW
        assert (CW - 1) + pos - 1 < bw * bh, "the flat run reaches past the box"
    else:
        assert bw == CW and bh >= L["halo_rows"], "the box covers the halo region"


XBUF_BYTES = 2 * 8 * 8 * 32 * 4   # the stacked kernel's epilogue shift buffers: 2 tiles x 8 warps x 8 lanes x 32 words


def check_stacked_layout(shape, L):
    """The stacked-tap kernel: halo segments of L = 128 + (S-1)*dw positions
    per filter row, A views of tap pairs 2*dw apart, filter stages of U slots
    of 64 fp16 rows, the epilogue's shift buffers, 2 x 128 accumulator columns."""
    N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw = shape
    assert K == 64 and sh == 1 and sw == 1 and 2 <= S <= 16 and dw <= 8
    U = (S + 1) // 2
    seg = 128 + (S - 1) * dw
    assert L["halo_cw"] == seg and L["halo_rows"] == R and L["positions"] == R * seg
    assert L["tile_px"] == 128 - dw, "valid outputs per tile"
    rows = L["chunk_slices"]
    assert rows >= 1 and rows * U * 32 <= 1024, "a column sums at most 1024 products per chunk"
    assert L["num_chunks"] * rows >= (C // 32) * R
    pos, plane = L["positions"], L["plane_bytes"]
    assert L["halo_bytes"] == 4 * plane and plane % 128 == 0 and plane >= 16 * pos
    # the furthest A row: segment R-1, the last slot's view ((S-1)*dw), row 127
    reach = (R - 1) * seg + (S - 1) * dw + 127
    assert reach < pos, f"an operand view reaches halo position {reach} of {pos}"
    assert 3 * plane + 16 * reach + 15 < L["halo_bytes"]
    assert 2 <= L["halo_stages"] <= 3
    assert L["off_out"] >= L["halo_stages"] * L["halo_bytes"], "shift buffers overlap the halo"
    assert L["off_out"] + XBUF_BYTES <= L["off_filter"], "shift buffers overlap the filter"
    assert L["off_filter"] % 1024 == 0
    assert L["filter_run"] == U and L["filter_stage_bytes"] == U * 64 * 64
    assert 1 <= L["filter_stages"] <= KMAX_FILTER_STAGES
    assert L["off_filter"] + L["filter_stages"] * L["filter_stage_bytes"] <= L["off_bar"]
    assert KHALO_BARRIER_WORDS * 8 <= L["bar_bytes"]
    assert L["off_bar"] + L["bar_bytes"] + 1024 <= L["smem_bytes"] <= KMAX_SMEM
    assert L["tmem_cols"] >= 2 * 128


PLAN_FORMS = [
    {}, dict(kernel_variant=1), dict(kernel_variant=2), dict(kernel_variant=2, halo_loads=1),
    dict(kernel_variant=2, halo_loads=2), dict(kernel_variant=3), dict(kernel_variant=3, block_n=64),
    dict(kernel_variant=3, block_n=256, halo_loads=1), dict(kernel_variant=2, tile_shape=2),
    dict(kernel_variant=3, tile_shape=2), dict(kernel_variant=2, block_n=32), dict(kernel_variant=2, block_n=256),
    dict(kernel_variant=4), dict(kernel_variant=4, tile_px=16), dict(kernel_variant=4, tile_px=176),
    dict(kernel_variant=4, tile_px=256), dict(kernel_variant=4, tile_px=64, filter_run=3),
    dict(kernel_variant=4, halo_loads=1), dict(kernel_variant=5), dict(kernel_variant=5, tile_px=128),
    dict(kernel_variant=5, tile_px=240, halo_loads=1), dict(max_chunk_slices=5), dict(kernel_variant=2, max_chunk_slices=7),
    dict(kernel_variant=6), dict(kernel_variant=6, max_chunk_slices=4),
    dict(halo_loads=3), dict(kernel_variant=2, halo_loads=3), dict(kernel_variant=3, halo_loads=3),
    dict(kernel_variant=2, tile_shape=2, halo_loads=3), dict(kernel_variant=3, block_n=64, halo_loads=3),
    dict(kernel_variant=4, halo_loads=3), dict(kernel_variant=4, tile_px=256, halo_loads=3),
    dict(kernel_variant=5, halo_loads=3), dict(kernel_variant=5, tile_px=128, halo_loads=3),
    dict(fused_filter=2), dict(kernel_variant=2, fused_filter=2), dict(kernel_variant=3, fused_filter=2),
    dict(kernel_variant=3, halo_loads=3, fused_filter=2), dict(fused_filter=3), dict(kernel_variant=3, fused_filter=3),
    dict(tile_shape=3), dict(tile_shape=3, kernel_variant=3), dict(tile_shape=3, kernel_variant=2, block_n=64),
    dict(tile_shape=3, kernel_variant=3, halo_loads=1), dict(tile_shape=3, kernel_variant=2, block_n=128),
    dict(tile_shape=3, kernel_variant=3, block_n=128),
]

SHAPES = [wl.shape_tuple() for wl in synth.WORKLOADS] + SMALL + TRANSPOSED_EXTRA + STACKED_SHAPES + [
    (1, 1024, 8, 8, 256, 3, 3, 1, 1, 1, 1, 1, 1), (2, 512, 7, 6, 64, 3, 3, 1, 1, 1, 1, 1, 1),
    (1, 1120, 6, 6, 416, 3, 3, 1, 1, 1, 1, 1, 1), (2, 32, 40, 40, 64, 5, 9, 2, 4, 1, 1, 2, 3)]


@pytest.fixture(scope="module")
def ext():
    import __graft_entry__
    __graft_entry__.build()
    import int8_implicit_gemm_gb300 as ext
    return ext


def _layout(ext, shape, opts):
    try:
        return ext.i8c_plan_layout(shape, 152, **opts)
    except ext.I8ConvError as e:
        if e.status == ext.I8C_ERR_UNSUPPORTED:
            return None
        raise


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_every_plan_form_stays_in_bounds(ext, shape):
    checked = 0
    for opts in PLAN_FORMS:
        L = _layout(ext, shape, opts)
        if L is None:
            continue
        check_layout(shape, L)
        checked += 1
    assert checked >= 2


@pytest.mark.parametrize("plant", ["positions", "plane_bytes", "off_bar", "off_staging", "tmem_cols", "off_out",
                                   "stacked_positions", "stacked_xbuf", "tma_box", "tma_slots"])
def test_planted_off_by_one_is_caught(ext, plant):
    """Each planted mistake shrinks one region by the smallest step the
    layout allows; the check must notice."""
    cases = {
        "positions": ((8, 256, 56, 56, 256, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=4), -1),
        "plane_bytes": ((32, 128, 112, 112, 256, 3, 3, 1, 1, 2, 2, 1, 1), {}, None),
        "off_bar": ((8, 32, 512, 512, 64, 5, 9, 2, 4, 1, 1, 2, 3), {}, None),
        "off_staging": ((2, 64, 13, 11, 64, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=2, halo_loads=1), None),
        "tmem_cols": ((64, 512, 28, 28, 512, 3, 3, 1, 1, 1, 1, 1, 1), {}, None),
        "off_out": ((8, 256, 56, 56, 256, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=4), None),
        "stacked_positions": ((8, 32, 512, 512, 64, 5, 9, 2, 4, 1, 1, 2, 3), dict(kernel_variant=6), None),
        "stacked_xbuf": ((8, 32, 512, 512, 64, 5, 9, 2, 4, 1, 1, 2, 3), dict(kernel_variant=6), None),
        "tma_box": ((8, 256, 56, 56, 256, 3, 3, 1, 1, 1, 1, 1, 1), dict(kernel_variant=4, halo_loads=3), None),
        "tma_slots": ((32, 128, 112, 112, 256, 3, 3, 1, 1, 2, 2, 1, 1), dict(kernel_variant=2, halo_loads=3), None),
    }
    shape, opts, _ = cases[plant]
    L = _layout(ext, shape, opts)
    check_layout(shape, L)                 # the real layout passes
    bad = dict(L)
    if plant == "positions":
        bad["positions"] -= 1
    elif plant == "plane_bytes":
        bad["plane_bytes"] = (16 * L["positions"] + 127) // 128 * 128 - 128
        bad["halo_bytes"] = 4 * bad["plane_bytes"]
    elif plant == "off_bar":   # barriers placed over the last 16 bytes of the filter stages
        bad["off_bar"] = L["off_filter"] + L["filter_stages"] * L["filter_stage_bytes"] - 16
    elif plant == "off_staging":
        bad["off_staging"] = L["halo_stages"] * L["halo_bytes"] - 16
    elif plant == "tmem_cols":
        bad["tmem_cols"] //= 2
    elif plant == "off_out":
        bad["off_out"] -= 1024
    elif plant == "stacked_positions":   # one halo position short
        bad["positions"] -= 1
    elif plant == "stacked_xbuf":        # shift buffers one row into the filter stages
        bad["off_out"] = L["off_filter"] - XBUF_BYTES + 128
    elif plant == "tma_box":             # a box one padded row short of the flat run
        bad["box_h"] -= 1
    elif plant == "tma_slots":           # int8 slots reaching one KB into the filter stages
        bad["off_x8"] += 1024
    with pytest.raises(AssertionError):
        check_layout(shape, bad)


def test_in_kernel_resident_filter_needs_a_resident_halo_plan(ext):
    """fused_filter = 2 (the kernel writes its resident filter into shared
    memory itself) is planned only where the halo kernel keeps the whole
    filter resident; elsewhere the planner refuses it on the host."""
    dilated = (8, 32, 512, 512, 64, 5, 9, 2, 4, 1, 1, 2, 3)      # 45 K-slices x 32 rows per CTA: resident
    wide = (32, 128, 112, 112, 256, 3, 3, 1, 1, 2, 2, 1, 1)      # 36 K-slices x 256 rows: streamed
    L = ext.i8c_plan_layout(dilated, 152, kernel_variant=3, fused_filter=2)
    check_layout(dilated, L)
    assert L["filter_stages"] * L["filter_run"] == 45
    for shape, opts in ((wide, dict(kernel_variant=2, fused_filter=2)),
                        (dilated, dict(kernel_variant=4, fused_filter=2)),
                        (dilated, dict(kernel_variant=6, fused_filter=2)),
                        (dilated, dict(kernel_variant=1, fused_filter=2))):
        with pytest.raises(ext.I8ConvError) as e:
            ext.i8c_plan_layout(shape, 152, **opts)
        assert e.value.status == ext.I8C_ERR_UNSUPPORTED, opts


def _random_shapes(seed, count):
    """Seeded convolution shapes across the planner's ranges: channel counts
    that are multiples of 32 (K also ragged), filters 1-9 taps a side,
    strides 1-4, dilations 1-4, paddings up to the filter's reach, images
    from a few pixels to a few hundred."""
    import random
    rng = random.Random(seed)
    out = []
    while len(out) < count:
        R, S = rng.randint(1, 9), rng.randint(1, 9)
        sh, sw = rng.choice([1, 1, 1, 2, 2, 3, 4]), rng.choice([1, 1, 1, 2, 2, 3, 4])
        dh, dw = rng.choice([1, 1, 2, 3, 4]), rng.choice([1, 1, 2, 3, 4])
        ph, pw = rng.randint(0, (R - 1) * dh), rng.randint(0, (S - 1) * dw)
        H, W = rng.randint(1, 160), rng.randint(1, 320)
        N = rng.randint(1, 8)
        C = 32 * rng.choice([1, 1, 2, 3, 4, 8, 16])
        K = rng.choice([32, 64, 96, 128, 160, 256, 512, 24, 200])
        shape = (N, C, H, W, K, R, S, ph, pw, sh, sw, dh, dw)
        P = (H + 2 * ph - dh * (R - 1) - 1) // sh + 1
        Q = (W + 2 * pw - dw * (S - 1) - 1) // sw + 1
        if P >= 1 and Q >= 1:
            out.append(shape)
    return out


@pytest.mark.parametrize("seed", [11, 12, 13, 14])
def test_random_shapes_every_plan_form_stays_in_bounds(ext, seed):
    """Seeded random shapes through every plan form: every layout the planner
    accepts passes the same bounds check as the fixed shapes (the planner
    may refuse a form for a shape; it must never hand a kernel a layout whose
    accesses leave their regions)."""
    accepted = 0
    for shape in _random_shapes(seed, 150):
        if ext.i8c_supported(shape) != ext.I8C_OK:
            continue
        for opts in PLAN_FORMS:
            L = _layout(ext, shape, opts)
            if L is None:
                continue
            check_layout(shape, L)
            accepted += 1
    assert accepted >= 1000
