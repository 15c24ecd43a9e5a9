"""The seeded input generator: lane-parallel xoshiro256** equals a scalar
restatement of the published algorithm, and the value mappings stay in range."""
import numpy as np

import synth

MASK = (1 << 64) - 1


def _scalar_splitmix(seed, count):
    out, x = [], seed & MASK
    for _ in range(count):
        x = (x + 0x9E3779B97F4A7C15) & MASK
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
        out.append(z ^ (z >> 31))
    return out


def _rotl(x, k):
    return ((x << k) | (x >> (64 - k))) & MASK


def _scalar_xoshiro(state, n):
    s = list(state)
    out = []
    for _ in range(n):
        out.append((_rotl((s[1] * 5) & MASK, 7) * 9) & MASK)
        t = (s[1] << 17) & MASK
        s[2] ^= s[0]; s[3] ^= s[1]; s[1] ^= s[2]; s[0] ^= s[3]; s[2] ^= t
        s[3] = _rotl(s[3], 45)
    return out


def test_lanes_match_scalar():
    seed, lanes = 12345, 8
    words = _scalar_splitmix(seed, 4 * lanes)
    g = synth.Xoshiro256ss(seed, lanes=lanes)
    got = g.next_u64(lanes * 5)
    for lane in range(lanes):
        want = _scalar_xoshiro(words[4 * lane: 4 * lane + 4], 5)
        assert [int(v) for v in got[lane::lanes]] == want


def test_value_ranges_and_determinism():
    a = synth.uniform_int8(1, 100000, -64, 63)
    assert a.min() == -64 and a.max() == 63
    assert np.array_equal(a, synth.uniform_int8(1, 100000, -64, 63))
    b = synth.normal_int8(2, 100000, 32.0)
    assert b.min() >= -128 and b.max() <= 127
    assert 28 < b.astype(np.float64).std() < 36


def test_workloads_table():
    assert len(synth.WORKLOADS) == 5
    for w in synth.WORKLOADS:
        assert w.C % 32 == 0 and w.K % 32 == 0


def test_uniform_f32_mapping_and_range():
    """uniform_f32 maps the top 24 bits of each draw onto [lo, hi) exactly as
    its docstring states, is deterministic per seed, and never reaches hi."""
    u = synth.Xoshiro256ss(77).next_u64(4096)
    want = (-0.5 + 1.5 * ((u >> np.uint64(40)).astype(np.float64) / float(1 << 24))).astype(np.float32)
    got = synth.uniform_f32(77, 4096, -0.5, 1.0)
    assert got.dtype == np.float32 and np.array_equal(got, want)
    assert np.array_equal(got, synth.uniform_f32(77, 4096, -0.5, 1.0))
    assert got.min() >= -0.5 and got.max() < 1.0


def test_f32_workload_is_the_trace_layer():
    w = synth.F32_WORKLOAD
    assert w.shape_tuple() == (8, 32, 512, 512, 64, 5, 9, 2, 4, 1, 1, 2, 3)
    assert abs(w.bound() - 1.0 / np.sqrt(32 * 5 * 9)) < 1e-15
    b = w.bias()
    assert b.shape == (64,) and np.all(np.abs(b) <= w.bound())
