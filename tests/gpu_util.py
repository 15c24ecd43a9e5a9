"""Shared helpers for the GPU parity tests: move seeded host data through the
C-ABI and bring results back.  The oracle's own layout helpers pack the
inputs and the oracle's results, so both sides read the same host buffers."""
from __future__ import annotations

import numpy as np

import oracle


def packed_inputs(x_nchw: np.ndarray, f_kcrs: np.ndarray):
    return oracle.nchw_to_ncxhwx32(x_nchw), oracle.kcrs_to_cxrskx32(f_kcrs)


def gpu_run(shape, x_nchw, f_kcrs, alpha, want_acc=True, **plan_kw):
    """Run the library on packed copies of x/f: (y, acc) as packed numpy arrays."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    xp, fp = packed_inputs(x_nchw, f_kcrs)
    xd = torch.from_numpy(xp).cuda()
    fd = torch.from_numpy(fp).cuda()
    plan = ext.Plan(shape, **plan_kw)
    N, K = shape[0], shape[4]
    P, Q = plan.info["P"], plan.info["Q"]
    y = torch.full((N, K // 32, P, Q, 32), 77, dtype=torch.int8, device="cuda")
    plan.run(xd, fd, y, alpha)
    acc = None
    if want_acc:
        acc = torch.full((N, K // 32, P, Q, 32), -7, dtype=torch.int32, device="cuda")
        plan.run_acc(xd, fd, acc)
    torch.cuda.synchronize()
    st = plan.status()
    assert st == 0, ext.status_string(st)
    out = y.cpu().numpy(), (acc.cpu().numpy() if acc is not None else None)
    plan.destroy()
    return out


def oracle_packed(shape, x_nchw, f_kcrs, alpha):
    """Oracle (y, acc) packed into the interleaved output layout."""
    orc = oracle.Oracle()
    y, acc = orc.conv2d_fprop(x_nchw, f_kcrs, shape, alpha)
    return oracle.nchw_to_ncxhwx32(y), oracle.nchw_to_ncxhwx32(acc)


def sample_points(shape, P, Q, count, seed):
    """Output coordinates (n, k, p, q): random ones plus borders, corners,
    GEMM tile boundaries and the last pixel."""
    N, K = shape[0], shape[4]
    rng = np.random.default_rng(seed)
    pts = [np.stack([rng.integers(0, N, count), rng.integers(0, K, count),
                     rng.integers(0, P, count), rng.integers(0, Q, count)], axis=1)]
    extra = []
    for n in {0, N - 1}:
        for k in {0, K - 1, min(31, K - 1), min(32, K - 1)}:
            for p in {0, 1, P // 2, P - 2 if P > 1 else 0, P - 1}:
                for q in {0, 1, Q // 2, Q - 2 if Q > 1 else 0, Q - 1}:
                    extra.append((n, k, p, q))
    PQ = P * Q
    for m in (127, 128, 129, 255, 256, N * PQ - 1):
        if m < N * PQ:
            n, pq = divmod(m, PQ)
            p, q = divmod(pq, Q)
            for k in (0, K - 1):
                extra.append((n, k, p, q))
    pts.append(np.array(extra, dtype=np.int64).reshape(-1, 4))
    return np.concatenate(pts).astype(np.int64)


def packed_index(shape, P, Q, pts):
    """Flat offsets of (n, k, p, q) in the interleaved NCxHWx<32> output."""
    K = shape[4]
    n, k, p, q = pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]
    return (((n * (K // 32) + k // 32) * P + p) * Q + q) * 32 + k % 32
