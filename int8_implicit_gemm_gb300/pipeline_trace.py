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
    the loop bookkeeping after them; per-CTA timeline (median, max in
    microseconds): entry to the MMA loop, the loop, loop end to exit, and
    the first entry to the last exit over all CTAs;
  - prod_* (halo kernel): producer thread 0's time from its halo stage being
    free to its arrival, from its arrival to the next stage being free, and
    its period per channel block, in microseconds; for the register-load
    producer also from its arrival to the next channel block's first load,
    the time to issue that block's loads, from their issue to the stage being free, from the
    stage being free to its stores done, and from the stores to its arrival
    (the fence and the arrive) (the *_cta1 keys: the same
    for CTA 1, a pair's rank 1; cta1_arrive_lag_us: how much later rank 1
    announces each halo stage than rank 0);
  - cb_interval_us: median and maximum time between consecutive halo
    acquisitions of the MMA warp.

  python -m int8_implicit_gemm_gb300.pipeline_trace n32c128h112k256r3s2 '{"num_ctas": 19}'

Plan options go in the JSON object; "prepacked": true traces prepacked runs
(the filter converted once by set_filter, then run_prepacked).
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
    prepacked = bool(opts.pop("prepacked", False))
    plan = ext.Plan(shape, debug_flags=2, **opts)
    if prepacked:  # the filter converted once, then the convolution alone, back to back
        plan.set_filter(sets[0][1])
    for i in range(runs):
        if prepacked:
            plan.run_prepacked(sets[i % nsets][0], sets[i % nsets][2], alpha)
        else:
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
        # per-CTA global-timer marks: kernel entry (8), MMA loop start (24)
        # and end (25), kernel exit (9)
        st, ls, le, en = tr[8][:512], tr[24][:512], tr[25][:512], tr[9][:512]
        ok = (st > 0) & (ls > 0) & (le > 0) & (en > 0)
        if ok.any():
            us = lambda v: round(float(v) / 1e3, 2)
            out["cta_span_us"] = [us(np.min(en[ok] - st[ok])), us(np.max(en[ok] - st[ok]))]
            out["entry_to_loop_us"] = [us(np.median(ls[ok] - st[ok])), us(np.max(ls[ok] - st[ok]))]
            out["loop_us"] = [us(np.median(le[ok] - ls[ok])), us(np.max(le[ok] - ls[ok]))]
            out["loop_to_exit_us"] = [us(np.median(en[ok] - le[ok])), us(np.max(en[ok] - le[ok]))]
            out["first_entry_to_last_exit_us"] = us(np.max(en[ok]) - np.min(st[ok]))
            out["entry_skew_us"] = us(np.max(st[ok]) - np.min(st[ok]))
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
        # producer thread 0 of CTA 0 and of CTA 1 (a pair's rank 1)
        for cta, suffix in ((0, ""), (1, "_cta1")):
            free, arrive = tr[16 + 2 * cta], tr[17 + 2 * cta]
            m = int(np.sum((free > 0) & (arrive > 0)))
            if m > 3:
                out["prod_free_to_arrive_us" + suffix] = round(float(np.median(arrive[1:m] - free[1:m])) / 1e3, 3)
                out["prod_arrive_to_next_free_us" + suffix] = round(
                    float(np.median(free[2:m] - arrive[1:m - 1])) / 1e3, 3)
                out["prod_period_us" + suffix] = round(float(np.median(np.diff(arrive[1:m]))) / 1e3, 3)
            # direct register-load producer: loads issued, stores done
            issued, stored = tr[28 + cta], tr[26 + cta]
            k = int(np.sum((issued > 0) & (stored > 0) & (free > 0) & (arrive > 0)))
            if k > 3:
                out["prod_issue_to_free_us" + suffix] = round(float(np.median(free[1:k] - issued[1:k])) / 1e3, 3)
                out["prod_free_to_stored_us" + suffix] = round(float(np.median(stored[1:k] - free[1:k])) / 1e3, 3)
                out["prod_stored_to_arrive_us" + suffix] = round(float(np.median(arrive[1:k] - stored[1:k])) / 1e3, 3)
                before = tr[30 + cta]  # before the first load of the channel block
                if int(np.sum(before > 0)) > k - 1:
                    out["prod_arrive_to_before_loads_us" + suffix] = round(
                        float(np.median(before[2:k] - arrive[1:k - 1])) / 1e3, 3)
                    out["prod_loads_issue_us" + suffix] = round(float(np.median(issued[1:k] - before[1:k])) / 1e3, 3)
        if info["kernel_variant"] == 3:
            a0, a1 = tr[17], tr[19]
            m = int(min(np.sum(a0 > 0), np.sum(a1 > 0)))
            if m > 3:
                # how much later the pair's rank 1 announces the same halo stage
                out["cta1_arrive_lag_us"] = round(float(np.median(a1[1:m] - a0[1:m])) / 1e3, 3)
                # and how much later it sees the same stage freed by the MMA's commit
                f0, f1 = tr[16], tr[18]
                mf = int(min(np.sum(f0 > 0), np.sum(f1 > 0)))
                if mf > 3:
                    out["cta1_free_lag_us"] = round(float(np.median(f1[1:mf] - f0[1:mf])) / 1e3, 3)
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
