"""The multi-rank ring on one GPU: N ranks emulated in one process.

Each rank's kernels (ra_fwd_block per block pair, ra_merge_partials at the
end) run on a stream of its own; the key/value blocks move between the ranks'
buffers by device copies on a copy stream, ordered by events only (no kernel
waits on another).  The assembled result is checked against the fp64 oracle
on every row with the forward's tolerances, for both sequence layouts, causal
and not, D = 64 and 128, and the caller's key/value pieces must come back
unchanged (the ring receives into buffers of its own).  A world-size-1 NCCL
group runs the multi-process entry point end to end.
"""
import os
import socket

import pytest
import torch

from ring_chunked_attention_gb300.inputs import Workload, make_inputs
from ring_chunked_attention_gb300.ring import (RingSpec, ring_attention, shard, unshard,
                                               virtual_ring_attention)
from tests.parity import assert_parity, compare

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Hkv, S, D, causal, layout, world
    (1, 4, 2, 2048, 128, True, "contiguous", 4),
    (1, 4, 2, 2048, 128, True, "zigzag", 4),
    (2, 2, 2, 1024, 64, False, "contiguous", 2),
    (1, 4, 1, 2048, 64, True, "zigzag", 2),
    (1, 2, 2, 3072, 128, False, "zigzag", 3),
    (1, 8, 2, 4096, 128, True, "zigzag", 8),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[6]}-{'causal' if c[5] else 'full'}-D{c[4]}-N{c[7]}"
                                             for c in CASES])
def test_virtual_ring_matches_the_oracle(ralib, cuda_ok, oracle_mod, case):
    B, H, Hkv, S, D, causal, layout, world = case
    w = Workload("vring", B, H, Hkv, S, D, world, causal)
    q, k, v = make_inputs(w, seed=67)
    spec = RingSpec(world, B, H, Hkv, S, D, causal, layout)
    qs = [shard(q, spec, r).cuda() for r in range(world)]
    ks = [shard(k, spec, r).cuda() for r in range(world)]
    vs = [shard(v, spec, r).cuda() for r in range(world)]
    keep = [(a.clone(), b.clone()) for a, b in zip(ks, vs)]
    res = virtual_ring_attention(qs, ks, vs, causal=causal, layout=layout)
    torch.cuda.synchronize()
    assert ralib.ra_get_last_device_status() == ralib.RA_OK
    for (a, b), (ka, kb) in zip(zip(ks, vs), keep):
        assert torch.equal(a, ka) and torch.equal(b, kb)
    out = unshard([o for o, _ in res], spec)
    lse = unshard([l for _, l in res], spec, seq_dim=2)
    o_ref, l_ref = oracle_mod.attn_direct(q, k, v, causal, w.scale)
    assert_parity(compare(out, lse, o_ref, l_ref), f"virtual ring {case}")


def test_ring_entry_point_on_a_one_rank_nccl_group(ralib, cuda_ok, oracle_mod):
    """ring_attention through a torch.distributed NCCL group of one rank: no
    exchange, one block per query piece (zig-zag: three, merged)."""
    import torch.distributed as dist

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        w = Workload("ring1", 1, 4, 2, 1024, 128, 1, True)
        q, k, v = make_inputs(w, seed=71)
        o_ref, l_ref = oracle_mod.attn_direct(q, k, v, True, w.scale)
        for layout in ("contiguous", "zigzag"):
            spec = RingSpec(1, 1, 4, 2, 1024, 128, True, layout)
            out, lse = ring_attention(shard(q, spec, 0).cuda(), shard(k, spec, 0).cuda(),
                                      shard(v, spec, 0).cuda(), causal=True, layout=layout)
            torch.cuda.synchronize()
            out = unshard([out], spec)
            lse = unshard([lse], spec, seq_dim=2)
            assert_parity(compare(out, lse, o_ref, l_ref), f"one-rank ring {layout}")
    finally:
        dist.destroy_process_group()
