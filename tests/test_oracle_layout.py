"""The oracle's layout helpers against the interleaved layouts' offset formulas,
element by element on small tensors (NCxHWx<32> and CxRSKx<32>, the layouts
named in page 1's CUTLASS configuration)."""
import numpy as np

import oracle


def test_ncxhwx32_offsets():
    rng = np.random.default_rng(1)
    N, C, H, W = 2, 64, 3, 5
    a = rng.integers(-128, 128, size=(N, C, H, W)).astype(np.int8)
    packed = oracle.nchw_to_ncxhwx32(a).reshape(-1)
    for n in range(N):
        for c in range(C):
            for h in range(H):
                for w in range(W):
                    off = (((n * (C // 32) + c // 32) * H + h) * W + w) * 32 + c % 32
                    assert packed[off] == a[n, c, h, w]
    assert np.array_equal(oracle.ncxhwx32_to_nchw(packed, N, C, H, W), a)


def test_cxrskx32_offsets():
    rng = np.random.default_rng(2)
    K, C, R, S = 3, 64, 2, 3
    f = rng.integers(-128, 128, size=(K, C, R, S)).astype(np.int8)
    packed = oracle.kcrs_to_cxrskx32(f).reshape(-1)
    for k in range(K):
        for c in range(C):
            for r in range(R):
                for s in range(S):
                    off = ((((c // 32) * R + r) * S + s) * K + k) * 32 + c % 32
                    assert packed[off] == f[k, c, r, s]
    assert np.array_equal(oracle.cxrskx32_to_kcrs(packed, K, C, R, S), f)
