"""Ring attention across ranks: sequence parallelism on top of libringattn.

The "Ring Attention" row of the mKernel overview page (chatgpz.de, table "Die
fünf verschmolzenen Kerne"): the sequence is sharded over the ranks of a ring.
At each of N steps a rank computes attention of its query block against the
key/value block it currently holds, while that block moves on to the next
rank and the previous rank's block arrives; N steps later every rank has
seen every block, and the per-block partial results are folded into the exact
result with the online-softmax (log-sum-exp) merge.

Here the exchange is driven by the host, one step at a time:

* ``RingRank.begin_step`` posts the send of the block held to rank r+1 and the
  receive of rank r-1's block into a second local buffer (torch.distributed
  point-to-point, NCCL on GPUs), so the copy runs while the kernels of the
  step compute on the current block;
* ``RingRank.compute_step`` launches ``ra_fwd_block`` once per (query piece,
  key/value piece) pair that holds an allowed key, writing a normalised
  partial (out, lse) into its slot;
* ``RingRank.end_step`` waits for the exchange and swaps the buffers;
* ``RingRank.finish`` folds each query piece's partials with
  ``ra_merge_partials``.

Every block the kernels read has first been received into this GPU's own
memory: no kernel is given a peer's pointer, and no multicast is used.  The
caller's k and v are never written (two buffers of the block's size are
allocated for the blocks in flight).

Sequence layouts (``layout``):

* ``"contiguous"``: the sequence of length S is cut into N chunks of C = S/N
  rows; rank r holds chunk r.  Local tensors are [B, C, heads, D].  Causal
  attention is unbalanced: rank r needs r+1 of the N blocks.
* ``"zigzag"``: the sequence is cut into 2N half-chunks of c = S/(2N) rows;
  rank r holds half-chunks r and 2N-1-r, so every rank has the same causal
  work.  Local tensors are [2, B, c, heads, D] (the two half-chunks stacked in
  front, each a contiguous [B, c, heads, D] block).  This balanced assignment
  is not on the pages; it is the usual companion of causal ring attention.

The compute calls go through an ``ops`` object; the default,
:class:`LibraryOps`, calls the library (there is no other product path).
Tests of the schedule on CPU ranks pass their own ops.
"""
from __future__ import annotations

from dataclasses import dataclass

__all__ = ["RingSpec", "RingRank", "LibraryOps", "DistTransport", "LocalRingTransport",
           "ring_attention", "virtual_ring_attention", "shard", "unshard", "block_plan"]


@dataclass(frozen=True)
class RingSpec:
    """Shape of one ring problem: the full sequence length S over N ranks."""
    world: int
    B: int
    H: int
    Hkv: int
    S: int
    D: int
    causal: bool
    layout: str = "contiguous"
    scale: float | None = None

    def __post_init__(self):
        if self.layout not in ("contiguous", "zigzag"):
            raise ValueError(f"unknown layout {self.layout!r}")
        pieces = self.world * (2 if self.layout == "zigzag" else 1)
        if self.world < 1 or self.S % pieces != 0:
            raise ValueError(f"S = {self.S} must split into {pieces} equal pieces")
        if self.H % self.Hkv != 0:
            raise ValueError("H must be a multiple of Hkv")

    @property
    def n_pieces(self) -> int:
        """Pieces of the sequence a rank holds (1 contiguous, 2 zig-zag)."""
        return 2 if self.layout == "zigzag" else 1

    @property
    def piece(self) -> int:
        """Rows per piece."""
        return self.S // (self.world * self.n_pieces)

    @property
    def softmax_scale(self) -> float:
        return self.D ** -0.5 if self.scale is None else float(self.scale)

    def positions(self, rank: int):
        """Global index of the first row of each piece rank ``rank`` holds."""
        if self.layout == "contiguous":
            return [rank * self.piece]
        return [rank * self.piece, (2 * self.world - 1 - rank) * self.piece]


def block_plan(spec: RingSpec, rank: int):
    """The ring schedule of one rank: for each step t, the rank j = (rank - t)
    mod N whose block is held, and the (query piece, key piece, q_pos0,
    k_pos0) pairs computed, with the partial slot each one fills.  A pair whose
    keys all lie after its last query (causal) is left out.  Returns
    (steps, parts_per_query_piece) with steps[t] = (j, [(qi, ki, q_pos0,
    k_pos0, slot), ...])."""
    L = spec.piece
    qpos = spec.positions(rank)
    counts = [0] * spec.n_pieces
    steps = []
    for t in range(spec.world):
        j = (rank - t) % spec.world  # the block rank j started with, received at step t
        pairs = []
        for qi, qp in enumerate(qpos):
            for ki, kp in enumerate(spec.positions(j)):
                if spec.causal and kp > qp + L - 1:
                    continue  # every key after every query row of the piece
                pairs.append((qi, ki, qp, kp, counts[qi]))
                counts[qi] += 1
        steps.append((j, pairs))
    return steps, counts


# ---------------------------------------------------------------- layouts
def shard(x, spec: RingSpec, rank: int):
    """Rank ``rank``'s piece(s) of a full-sequence tensor ``x`` [B, S, heads,
    D]: [B, C, heads, D] (contiguous) or [2, B, c, heads, D] (zig-zag)."""
    import torch

    L = spec.piece
    parts = [x[:, p:p + L] for p in spec.positions(rank)]
    if spec.layout == "contiguous":
        return parts[0].contiguous()
    return torch.stack(parts).contiguous()


def unshard(pieces, spec: RingSpec, seq_dim: int = 1):
    """Inverse of :func:`shard` over all ranks: ``pieces[r]`` is rank r's
    local tensor; returns the full-sequence tensor.  ``seq_dim`` is the
    sequence axis of one piece (1 for [B, S, heads, D], 2 for lse [B, H, S])."""
    import torch

    L = spec.piece
    order = {}
    for r, x in enumerate(pieces):
        ps = [x] if spec.layout == "contiguous" else [x[0], x[1]]
        for p, piece in zip(spec.positions(r), ps):
            order[p] = piece
    return torch.cat([order[p] for p in sorted(order)], dim=seq_dim)


# ------------------------------------------------------------------ compute
class LibraryOps:
    """The product compute path: libringattn's block step and merge."""

    def __init__(self, stream=None):
        self.stream = stream

    def empty_parts(self, n, B, L, H, D, like):
        import torch

        return (torch.empty((n, B, L, H, D), dtype=torch.bfloat16, device=like.device),
                torch.empty((n, B, H, L), dtype=torch.float32, device=like.device))

    def empty_out(self, shape_o, shape_l, like):
        import torch

        return (torch.empty(shape_o, dtype=torch.bfloat16, device=like.device),
                torch.empty(shape_l, dtype=torch.float32, device=like.device))

    def block(self, q, k, v, q_pos0, k_pos0, causal, scale, out, lse):
        from . import ra_fwd_block

        ra_fwd_block(q, k, v, q_pos0=q_pos0, k_pos0=k_pos0, causal=causal, scale=scale, out=out,
                     lse=lse, stream=self.stream)

    def merge(self, o_parts, lse_parts, out, lse):
        from . import ra_merge_partials

        ra_merge_partials(o_parts, lse_parts, out=out, lse=lse, stream=self.stream)


# -------------------------------------------------------------- transports
class DistTransport:
    """Point-to-point exchange over a torch.distributed process group: rank r
    sends to r+1 and receives from r-1 (NCCL for CUDA tensors, gloo for CPU
    ones).  bf16 blocks travel as int16 views (a byte copy either way)."""

    def __init__(self, group=None):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    @staticmethod
    def _wire(t):
        import torch

        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t

    def post(self, send, recv):
        dist = self.dist
        nxt = (self.rank + 1) % self.world
        prv = (self.rank - 1) % self.world
        if self.group is not None:
            nxt = dist.get_global_rank(self.group, nxt)
            prv = dist.get_global_rank(self.group, prv)
        ops = []
        for s, r in zip(send, recv):
            ops.append(dist.P2POp(dist.isend, self._wire(s), nxt, self.group))
            ops.append(dist.P2POp(dist.irecv, self._wire(r), prv, self.group))
        return dist.batch_isend_irecv(ops)

    def wait(self, handle):
        for w in handle:
            w.wait()


class LocalRingTransport:
    """N ranks emulated in one process on one GPU: rank r's receive buffers
    are filled by device-to-device copies of rank r-1's send buffers, issued
    on one copy stream once every rank has posted its step.  Each copy waits
    for an event that marks the end of the receiving rank's previous step (the
    buffer it overwrites was read there); each rank's next step waits for an
    event recorded after the copies.  Nothing spins on the GPU: the ordering
    is stream order and events only."""

    def __init__(self, world, device):
        import torch

        self.world = world
        self.copy_stream = torch.cuda.Stream(device=device)
        self.posts = {}

    def endpoint(self, rank, stream):
        return _LocalEndpoint(self, rank, stream)

    def _post(self, rank, send, recv, ready):
        import torch

        self.posts[rank] = (send, recv, ready)
        if len(self.posts) < self.world:
            return None
        cs = self.copy_stream
        for r in range(self.world):
            cs.wait_event(self.posts[r][2])
        with torch.cuda.stream(cs):
            for r in range(self.world):
                src = self.posts[(r - 1) % self.world][0]
                dst = self.posts[r][1]
                for s, d in zip(src, dst):
                    d.copy_(s, non_blocking=True)
        done = torch.cuda.Event()
        done.record(cs)
        self.posts = {}
        return done


class _LocalEndpoint:
    def __init__(self, hub, rank, stream):
        self.hub, self.rank, self.stream = hub, rank, stream
        self._done = None

    def post(self, send, recv):
        import torch

        ready = torch.cuda.Event()
        ready.record(self.stream)  # this rank's earlier reads of the receive buffers
        done = self.hub._post(self.rank, send, recv, ready)
        if done is not None:
            self.hub.last_done = done
        return self.hub

    def wait(self, hub):
        self.stream.wait_event(hub.last_done)


# ------------------------------------------------------------------- a rank
class RingRank:
    """One rank's side of the ring: its query piece(s), the key/value block in
    hand and the next one arriving, and the partial results."""

    def __init__(self, spec: RingSpec, rank: int, q, k, v, transport, ops=None):
        self.spec, self.rank = spec, rank
        self.ops = ops if ops is not None else LibraryOps()
        self.transport = transport
        L, n = spec.piece, spec.n_pieces
        lead = (2,) if spec.layout == "zigzag" else ()
        want_q = lead + (spec.B, L, spec.H, spec.D)
        want_kv = lead + (spec.B, L, spec.Hkv, spec.D)
        for t, name, want in ((q, "q", want_q), (k, "k", want_kv), (v, "v", want_kv)):
            if tuple(t.shape) != want:
                raise ValueError(f"{name} must have shape {want} on rank {rank}, got {tuple(t.shape)}")
        self.q = q
        self.plan, counts = block_plan(spec, rank)
        self.parts = [self.ops.empty_parts(c, spec.B, L, spec.H, spec.D, q) if c > 1 else None
                      for c in counts]
        self.out, self.lse = self.ops.empty_out(lead + (spec.B, L, spec.H, spec.D),
                                                lead + (spec.B, spec.H, L), q)
        self.counts = counts
        # the block in hand (the caller's k, v first, never written) and the
        # two buffers the later blocks arrive in
        self.cur = (k, v)
        self.bufs = [(k.new_empty(k.shape), v.new_empty(v.shape)) for _ in range(2 if spec.world > 1 else 0)]
        self.nxt = self.bufs[0] if self.bufs else None
        self._handle = None

    def _piece(self, x, i):
        return x if self.spec.layout == "contiguous" else x[i]

    def begin_step(self, t):
        if t + 1 < self.spec.world:
            self._handle = self.transport.post(self.cur, self.nxt)

    def compute_step(self, t):
        spec = self.spec
        _, pairs = self.plan[t]
        k, v = self.cur
        for qi, ki, qp, kp, slot in pairs:
            if self.counts[qi] == 1:  # the piece's only partial is its result
                o, l = self._piece(self.out, qi), self._piece(self.lse, qi)
            else:
                o, l = self.parts[qi][0][slot], self.parts[qi][1][slot]
            self.ops.block(self._piece(self.q, qi), self._piece(k, ki), self._piece(v, ki), qp, kp,
                           spec.causal, spec.softmax_scale, o, l)

    def end_step(self, t):
        if t + 1 < self.spec.world:
            self.transport.wait(self._handle)
            self._handle = None
            # the block just received is in hand; the next one goes to the
            # other buffer (the caller's k, v are never a receive target)
            arrived = self.nxt
            self.nxt = self.bufs[1] if arrived is self.bufs[0] else self.bufs[0]
            self.cur = arrived

    def finish(self):
        for i, c in enumerate(self.counts):
            if c > 1:
                self.ops.merge(self.parts[i][0], self.parts[i][1], self._piece(self.out, i),
                               self._piece(self.lse, i))
        return self.out, self.lse

    def run(self):
        for t in range(self.spec.world):
            self.begin_step(t)
            self.compute_step(t)
            self.end_step(t)
        return self.finish()


def ring_attention(q, k, v, *, causal: bool, layout: str = "contiguous", scale=None, group=None,
                   ops=None, S=None):
    """This rank's part of ring attention over a torch.distributed group.
    ``q`` / ``k`` / ``v`` are the rank's local pieces (see the module notes on
    layouts); returns the rank's (out, lse) pieces in the same layout (lse
    [B, H, C] or [2, B, H, c]).  ``S`` is the full sequence length (default:
    world x the local rows)."""
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        world, rank = dist.get_world_size(group), dist.get_rank(group)
    else:  # no process group: a ring of one rank (nothing is exchanged)
        world, rank = 1, 0
    zig = layout == "zigzag"
    B, L, H, D = tuple(q.shape[1:] if zig else q.shape)
    Hkv = k.shape[-2]
    spec = RingSpec(world, B, H, Hkv, S or world * L * (2 if zig else 1), D, causal, layout, scale)
    transport = DistTransport(group) if world > 1 else None
    return RingRank(spec, rank, q, k, v, transport, ops).run()


def virtual_ring_attention(qs, ks, vs, *, causal: bool, layout: str = "contiguous", scale=None):
    """N ranks of :func:`ring_attention` emulated in one process on one GPU:
    ``qs[r]``, ``ks[r]``, ``vs[r]`` are rank r's local pieces.  Each rank's
    kernels run on a stream of its own; the blocks move by device copies on a
    copy stream (:class:`LocalRingTransport`).  Returns the list of per-rank
    (out, lse)."""
    import torch

    world = len(qs)
    zig = layout == "zigzag"
    B, L, H, D = tuple(qs[0].shape[1:] if zig else qs[0].shape)
    spec = RingSpec(world, B, H, ks[0].shape[-2], world * L * (2 if zig else 1), D, causal, layout,
                    scale)
    dev = qs[0].device
    hub = LocalRingTransport(world, dev)
    streams = [torch.cuda.Stream(device=dev) for _ in range(world)]
    cur = torch.cuda.current_stream(dev)
    for s in streams:
        s.wait_stream(cur)
    ranks = [RingRank(spec, r, qs[r], ks[r], vs[r], hub.endpoint(r, streams[r]),
                      LibraryOps(stream=streams[r])) for r in range(world)]
    for t in range(world):
        for r in range(world):
            with torch.cuda.stream(streams[r]):
                ranks[r].begin_step(t)
        for r in range(world):
            with torch.cuda.stream(streams[r]):
                ranks[r].compute_step(t)
        for r in range(world):
            with torch.cuda.stream(streams[r]):
                ranks[r].end_step(t)
    res = []
    for r in range(world):
        with torch.cuda.stream(streams[r]):
            res.append(ranks[r].finish())
    for s in streams:
        cur.wait_stream(s)
    return res
