"""The multi-rank ring schedule on CPU ranks (gloo), checked against the oracle.

Each rank holds its piece(s) of the sequence (contiguous chunks, or the
zig-zag pair of half-chunks), passes its key/value block to the next rank at
every step over gloo point-to-point, computes each step's partials with the
oracle's block function and folds them with the oracle's merge (the compute
calls are passed in as ``ops``; the product path uses the library's kernels
instead).  The assembled result must equal the oracle's direct definition on
every row: that pins the ring order, the global positions of every piece, the
causal skipping and the fold.  No GPU is involved.
"""
import itertools
import os
import socket

import numpy as np
import pytest
import torch

from ring_chunked_attention_gb300.inputs import Workload, make_inputs
from ring_chunked_attention_gb300.ring import RingSpec, block_plan, shard, unshard

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """Compute calls of the ring on the CPU oracle (fp64 partials)."""

    def __init__(self, oracle):
        self.oracle = oracle

    def empty_parts(self, n, B, L, H, D, like):
        return np.empty((n, B, L, H, D)), np.empty((n, B, H, L))

    def empty_out(self, shape_o, shape_l, like):
        return np.empty(shape_o), np.empty(shape_l)

    def block(self, q, k, v, q_pos0, k_pos0, causal, scale, out, lse):
        o, l = self.oracle.attn_block(q, k, v, q_pos0, k_pos0, causal, scale)
        out[...] = o
        lse[...] = l

    def merge(self, o_parts, lse_parts, out, lse):
        o, l = self.oracle.merge(o_parts, lse_parts)
        out[...] = o
        lse[...] = l


def _rank_main(rank, world, port, out_dir, case):
    import sys

    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from ring_chunked_attention_gb300.ring import ring_attention

    B, H, Hkv, S, D, causal, layout = case
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    w = Workload("ring", B, H, Hkv, S, D, world, causal)
    q, k, v = make_inputs(w, seed=61)
    spec = RingSpec(world, B, H, Hkv, S, D, causal, layout)
    out, lse = ring_attention(shard(q, spec, rank), shard(k, spec, rank), shard(v, spec, rank),
                              causal=causal, layout=layout, ops=OracleOps(oracle))
    np.save(os.path.join(out_dir, f"out{rank}.npy"), out)
    np.save(os.path.join(out_dir, f"lse{rank}.npy"), lse)
    dist.barrier()
    dist.destroy_process_group()


CASES = [
    # B, H, Hkv, S, D, causal, layout ; world
    ((1, 4, 2, 512, 64, True, "contiguous"), 2),
    ((1, 4, 2, 512, 64, False, "contiguous"), 2),
    ((1, 4, 2, 512, 64, True, "zigzag"), 2),
    ((2, 2, 1, 1024, 32, True, "zigzag"), 4),
    ((1, 2, 2, 768, 32, True, "contiguous"), 3),
    ((1, 2, 1, 768, 32, False, "zigzag"), 3),
]


@pytest.mark.parametrize("case,world", CASES, ids=[f"{c[6]}-{'causal' if c[5] else 'full'}-N{n}"
                                                   for c, n in CASES])
def test_ring_over_gloo_ranks_equals_the_definition(tmp_path, oracle_mod, case, world):
    import torch.multiprocessing as mp

    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), case), nprocs=world,
                       join=True, start_method="spawn")
    B, H, Hkv, S, D, causal, layout = case
    spec = RingSpec(world, B, H, Hkv, S, D, causal, layout)
    outs = [torch.from_numpy(np.load(tmp_path / f"out{r}.npy")) for r in range(world)]
    lses = [torch.from_numpy(np.load(tmp_path / f"lse{r}.npy")) for r in range(world)]
    out = unshard(outs, spec).numpy()
    lse = unshard(lses, spec, seq_dim=2).numpy()
    q, k, v = make_inputs(Workload("ring", B, H, Hkv, S, D, world, causal), seed=61)
    o_ref, l_ref = oracle_mod.attn_direct(q, k, v, causal, D ** -0.5)
    assert np.abs(out - o_ref).max() <= 1e-12
    assert np.abs(lse - l_ref).max() <= 1e-12 * max(1.0, np.abs(l_ref).max())


# ------------------------------------------------------------- the plan alone
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("causal", [True, False])
def test_block_plan_covers_each_allowed_key_once(world, layout, causal):
    """Over the N steps, every key row a query piece may attend to lies in
    exactly one computed block, and no computed block lies wholly in a causal
    piece's future; at step t the block in hand is rank (r - t) mod N's."""
    L = 128
    spec = RingSpec(world, 1, 1, 1, L * world * (2 if layout == "zigzag" else 1), 64, causal, layout)
    for r in range(world):
        steps, counts = block_plan(spec, r)
        assert [j for j, _ in steps] == [(r - t) % world for t in range(world)]
        for qi, qp in enumerate(spec.positions(r)):
            seen = []
            for t, (j, pairs) in enumerate(steps):
                for pqi, ki, pqp, kp, slot in pairs:
                    if pqi != qi:
                        continue
                    assert pqp == qp and kp == spec.positions(j)[ki]
                    assert not (causal and kp > qp + L - 1)
                    seen.extend(range(kp, kp + L))
            # every key some row of the piece may attend to (causal: up to the
            # piece's last row; the diagonal block is masked inside the
            # kernel), each in exactly one block
            allowed = set(range(0, qp + L)) if causal else set(range(spec.S))
            assert len(seen) == len(set(seen))
            assert set(seen) == allowed
            slots = sorted(s for _, pairs in steps for pqi, _, _, _, s in pairs if pqi == qi)
            assert slots == list(range(counts[qi]))


@pytest.mark.parametrize("world", [2, 4, 8])
def test_zigzag_balances_causal_work(world):
    """Causal work per rank, in (query, key) pairs: contiguous chunks give rank
    r about (r + 1/2) C^2 pairs, the zig-zag pair of half-chunks gives every
    rank the same."""
    L = 128

    def pairs_of(spec, r):
        total = 0
        for _, pairs in block_plan(spec, r)[0]:
            for _, _, qp, kp, _ in pairs:
                for s, t in itertools.product(range(qp, qp + L, 16), range(kp, kp + L, 16)):
                    total += t <= s
        return total

    zz = RingSpec(world, 1, 1, 1, 2 * L * world, 64, True, "zigzag")
    work = [pairs_of(zz, r) for r in range(world)]
    assert max(work) == min(work)
    cont = RingSpec(world, 1, 1, 1, 2 * L * world, 64, True, "contiguous")
    cw = [pairs_of(cont, r) for r in range(world)]
    assert cw == sorted(cw) and cw[-1] > 2 * cw[0]


def test_shard_and_unshard_are_inverse():
    x = torch.arange(2 * 1024 * 3 * 4, dtype=torch.float32).reshape(2, 1024, 3, 4)
    for layout, world in (("contiguous", 4), ("zigzag", 4), ("zigzag", 2)):
        spec = RingSpec(world, 2, 3, 3, 1024, 4, True, layout)
        pieces = [shard(x, spec, r) for r in range(world)]
        assert torch.equal(unshard(pieces, spec), x)
        if layout == "zigzag":
            p0 = pieces[0]
            assert torch.equal(p0[0], x[:, :spec.piece])
            assert torch.equal(p0[1], x[:, -spec.piece:])
