"""Pipeline-trace summary of CTA 0 of one convolution launch.

Needs the pipeline-analysis build of the library (``python
int8_implicit_gemm_gb300/build_lib.py --pipeline-trace``); rebuild without the
flag afterwards.  Runs a workload a few times on rotating random inputs (more
bytes than L2), with the plan's trace buffer enabled, and prints one JSON line
per run configuration:

  - cycles / per_slice: the MMA warp's loop on CTA 0, in SM cycles, and per
    K-slice (32 input channels of one filter tap);
  - stall_h / stall_b / stall_acc: cycles the MMA warp spent in its waits for
    halos, filter stages and free accumulator buffers (each including the
    wait's fixed cost); nr_*: how many of those waits found the phase still
    open (halo kernel);
  - issue / post (transposed tiles): cycles inside the MMA issue blocks and in
    the loop bookkeeping after them;
  - prod_* (halo kernel): producer thread 0's time from its halo stage being
    free to its arrival, from its arrival to the next stage being free, and
    its period per channel block, in microseconds;
  - cb_interval_us: median and maximum time between consecutive halo
    acquisitions of the MMA warp.

  python -m int8_implicit_gemm_gb300.pipeline_trace n32c128h112k256r3s2 '{"num_ctas": 19}'
"""
from __future__ import annotations

import json
import math
import sys

L2_BYTES = 129 << 20


def trace_workload(shape, alpha, runs: int = 6, **opts) -> dict:
    import numpy as np
    import torch

    import int8_implicit_gemm_gb300 as ext
    P, Q = ext.i8c_output_size(shape)
    N, C, H, W, K, R, S = shape[:7]
    xb, fb, yb = N * C * H * W, K * C * R * S, N * K * P * Q
    nsets = max(1, min(64, math.ceil(2 * L2_BYTES / (xb + fb + yb))))
    g = torch.Generator(device="cuda").manual_seed(5)
    sets = [(torch.randint(-128, 128, (xb,), dtype=torch.int8, device="cuda", generator=g),
             torch.randint(-128, 128, (fb,), dtype=torch.int8, device="cuda", generator=g),
             torch.empty(yb, dtype=torch.int8, device="cuda")) for _ in range(nsets)]
    plan = ext.Plan(shape, debug_flags=2, **opts)
    for i in range(runs):
        plan.run(*sets[i % nsets], alpha)
    torch.cuda.synchronize()
    if plan.status() != 0:
        raise RuntimeError("a bounded wait ran out during the traced runs")
    tr = plan.trace().reshape(32, 512)
    info = plan.info
    out = {"kernel_variant": info["kernel_variant"], "filter_run": info["filter_run"],
           "chunk_slices": info["chunk_slices"]}
    t0, t1 = int(tr[0][0]), int(tr[0][1])
    if info["kernel_variant"] >= 4:
        slices = int(tr[4][0])
        out.update(cycles=t1 - t0, slices=slices, per_slice=round((t1 - t0) / max(1, slices), 1),
                   stall_acc=int(tr[4][1]), stall_b=int(tr[4][2]), stall_h=int(tr[4][3]), issue=int(tr[4][7]),
                   post=int(tr[4][8]), stall_h_first=int(tr[4][9]))
    elif info["kernel_variant"] >= 2:
        slices = int(tr[4][0])  # K-slices issued by CTA 0
        out.update(cycles=t1 - t0, slices=slices, per_slice=round((t1 - t0) / max(1, slices), 1),
                   stall_acc=int(tr[4][1]), stall_b=int(tr[4][2]), stall_h=int(tr[4][3]),
                   nr_acc=int(tr[4][4]), nr_b=int(tr[4][5]), nr_h=int(tr[4][6]))
        st, en = tr[8][:512], tr[9][:512]
        ok = (st > 0) & (en > 0)
        if ok.any():
            out["cta_span_us"] = [round(float(np.min(en[ok] - st[ok])) / 1e3, 2),
                                  round(float(np.max(en[ok] - st[ok])) / 1e3, 2)]
        free, arrive = tr[16], tr[17]
        m = int(np.sum((free > 0) & (arrive > 0)))
        if m > 3:
            out["prod_free_to_arrive_us"] = round(float(np.median(arrive[1:m] - free[1:m])) / 1e3, 3)
            out["prod_arrive_to_next_free_us"] = round(float(np.median(free[2:m] - arrive[1:m - 1])) / 1e3, 3)
            out["prod_period_us"] = round(float(np.median(np.diff(arrive[1:m]))) / 1e3, 3)
        acq = tr[20]
        n = int(np.sum(acq > 0))
        if n > 2:
            d = np.diff(acq[:n]) / 1e3
            out["cb_interval_us"] = [round(float(np.median(d)), 3), round(float(np.max(d)), 3)]
    plan.destroy()
    return out


def main(argv) -> None:
    import os
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import synth
    name = argv[1] if len(argv) > 1 else "n8c256h56k256r3s1"
    opts = json.loads(argv[2]) if len(argv) > 2 else {}
    wl = synth.WORKLOADS_BY_NAME[name]
    res = trace_workload(wl.shape_tuple(), wl.alpha, **opts)
    print(json.dumps({"workload": name, "options": opts, **res}), flush=True)


if __name__ == "__main__":
    main(sys.argv)
