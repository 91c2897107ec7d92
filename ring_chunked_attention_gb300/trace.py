"""Per-role cycle breakdown of the forward kernel, from the traced build.

Run with the traced library selected (``RA_TRACE=1``; built by
``python -m ring_chunked_attention_gb300.build --trace``):

    RA_TRACE=1 python -m ring_chunked_attention_gb300.trace --workload gqa_s16384
    RA_TRACE=1 python -m ring_chunked_attention_gb300.trace --workload d64_s32768 --pairing 2

It launches ``ra_fwd`` on the workload's seeded inputs (three launches, the
last one counted), reads the counters with ``ra_trace_read`` and prints, per
key/value step of one CTA (both query slots), where the MMA warp, the softmax
warps of each slot and the producer thread spend their cycles.  ``--pairing``
forces paired query tiles (1) or one query tile per item (2), as
``ra_set_item_pairing`` does.  The counting itself lengthens the launch by
about a tenth; compare shapes, not absolutes.
"""
from __future__ import annotations

import argparse
import os
import sys

# counter slots per CTA (see ra_internal.h)
MMA = {"P waits": 0, "PV issue": 1, "V waits": 2, "S issue": 3, "late K waits": 6,
       "item starts": 7, "step top": 14, "closing commits": 15}
MMA_STEPS, MMA_TOTAL, MMA_FIRST_V, MMA_ITEMS = 4, 5, 24, 25
MMA_ITEM = {"Q waits": 26, "waits for the previous item's last PV": 27}
SOFTMAX = {"S waits": 0, "S to P hand-off": 1, "after the hand-off": 2}
SOFTMAX_TILES, SOFTMAX_EPI, SOFTMAX_ITEMS = 3, 4, 5
PRODUCER = {"K-stage waits": 28, "V-stage waits": 29}
PRODUCER_Q = 30


def summarize(counters):
    """Dict of per-step / per-tile / per-item figures from an int64 tensor
    [ctas, 32] of one launch's counters."""
    c = counters.double()
    steps = float(c[:, MMA_STEPS].sum())
    items = float(c[:, MMA_ITEMS].sum())
    out = {"ctas": int(c.shape[0]), "steps per CTA": steps / c.shape[0],
           "cycles per step": float(c[:, MMA_TOTAL].sum()) / steps if steps else 0.0}
    for name, i in MMA.items():
        out[f"MMA warp: {name} per step"] = float(c[:, i].sum()) / steps if steps else 0.0
    for slot, base in ((0, 8), (1, 16)):
        tiles = float(c[:, base + SOFTMAX_TILES].sum())
        if not tiles:
            continue
        for name, i in SOFTMAX.items():
            out[f"softmax slot {slot}: {name} per tile"] = float(c[:, base + i].sum()) / tiles
        n_epi = float(c[:, base + SOFTMAX_ITEMS].sum())
        if n_epi:
            out[f"softmax slot {slot}: epilogue per item"] = float(c[:, base + SOFTMAX_EPI].sum()) / n_epi
    for name, i in PRODUCER.items():
        out[f"producer: {name} per step"] = float(c[:, i].sum()) / steps if steps else 0.0
    if items:
        out["producer: Q-slot waits per item"] = float(c[:, PRODUCER_Q].sum()) / items
        out["MMA warp: V waits at an item's first step, per item"] = float(c[:, MMA_FIRST_V].sum()) / items
        for name, i in MMA_ITEM.items():
            out[f"MMA warp: item start, {name}, per item"] = float(c[:, i].sum()) / items
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="gqa_s16384")
    ap.add_argument("--pairing", type=int, default=0, choices=(0, 1, 2),
                    help="0 automatic, 1 paired query tiles, 2 one query tile per item")
    args = ap.parse_args(argv)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import torch

    import ring_chunked_attention_gb300 as ra
    from ring_chunked_attention_gb300.inputs import WORKLOADS, make_inputs

    if not ra.ra_trace_build():
        print("the loaded library is not the traced build: set RA_TRACE=1 and build it with "
              "`python -m ring_chunked_attention_gb300.build --trace`", file=sys.stderr)
        return 2
    w = WORKLOADS[args.workload]
    q, k, v = (t.cuda() for t in make_inputs(w))
    ra.ra_set_item_pairing(args.pairing)
    try:
        for _ in range(3):
            ra.ra_fwd(q, k, v, P=w.P, causal=w.causal)
        torch.cuda.synchronize()
    finally:
        ra.ra_set_item_pairing(0)
    status = ra.ra_get_last_device_status()
    ctas = min(torch.cuda.get_device_properties(0).multi_processor_count, 1024)
    res = summarize(ra.ra_trace_read(ctas))
    print(f"{w.name} (pairing {args.pairing}): status {ra.ra_status_string(status)}")
    for key, val in res.items():
        print(f"  {key}: {val:,.0f}" if isinstance(val, float) else f"  {key}: {val}")
    return 0 if status == ra.RA_OK else 1


if __name__ == "__main__":
    sys.exit(main())
