"""Query-sharded KPool indexer: one process per GPU, each scoring a share of
the query rows.

The indexer partitions by query rows: a query needs only the pooled keys of
its own document's causal prefix (Megatron-LM PR "GLM5.3 Flash (KDA + mHC +
KPool DSA) support + FP8", Changes section 3; its context-parallel layout is
a zigzag split of the sequence, and the SkyRL PR "GLM-5.3-Flash (glm5_next)
Megatron support", commit "k-pool indexer", gathers the gate score across
context-parallel ranks).  Two layouts:

* one long sequence -- zigzag: the sequence is cut into 2W blocks on pool
  boundaries and rank r holds blocks r and 2W-1-r, so every rank gets the
  same share of the causal triangle.  A rank holds the q, k, gate and w rows
  of its blocks only; it compresses the pools of its own blocks, and one
  all-gather of pooled keys gives every rank the whole sequence's pooled keys
  (queries of a late block score pools of every earlier block).  Its queries
  then run as positioned queries (kpool_score_topk_at) over those pooled
  keys, and kpool_expand_indices_at writes global token indices.
* packed documents -- whole documents: contiguous runs of documents, cut so
  that each rank's causal work (sum of L_d^2) is close to 1/W of the total.
  A document's queries see only its own keys, so nothing is exchanged; the
  expansion is given the documents' global starts, so token indices are
  global here too.

Every rank can derive every rank's plan from (T, cu_seqlens, W, kpool), so
the exchange needs no size negotiation.  The arithmetic runs in the CUDA
library (`DeviceOps`); this module only plans shards, moves pooled keys and
places rows.  `ShardedIndexer` takes its operations as an object so that the
same plan and bookkeeping can be driven by another implementation of the
four operations (the tests drive it on CPU ranks).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch


@dataclass(frozen=True)
class Segment:
    """A contiguous range [start, end) of global token rows held by one rank,
    inside document `doc` (global start `doc_start`, first global pool
    `pool_base`).  `start - doc_start` is a multiple of kpool."""
    start: int
    end: int
    doc: int
    doc_start: int
    pool_base: int

    @property
    def rows(self) -> int:
        return self.end - self.start

    def pools(self, kpool: int) -> int:
        """Complete pools whose tokens all lie in the segment."""
        return (self.end - self.start) // kpool

    def first_pool(self, kpool: int) -> int:
        return self.pool_base + (self.start - self.doc_start) // kpool


@dataclass(frozen=True)
class ShardPlan:
    rank: int
    world: int
    kpool: int
    T: int
    P_total: int
    layout: str                      # "zigzag" or "documents"
    segments: tuple                  # this rank's segments, in local row order
    all_segments: tuple              # every rank's segments (tuple per rank)

    @property
    def exchange(self) -> bool:
        """Pooled keys must be gathered from the other ranks."""
        return self.layout == "zigzag" and self.world > 1

    @property
    def local_rows(self) -> int:
        return sum(s.rows for s in self.segments)

    def local_pools(self, rank: Optional[int] = None) -> int:
        segs = self.segments if rank is None else self.all_segments[rank]
        return sum(s.pools(self.kpool) for s in segs)

    def row_offsets(self) -> List[int]:
        """Local row offset of each of this rank's segments."""
        out, o = [], 0
        for s in self.segments:
            out.append(o)
            o += s.rows
        return out

    def local_row_index(self) -> torch.Tensor:
        """Global token row of each local row (int64)."""
        if not self.segments:
            return torch.zeros(0, dtype=torch.int64)
        return torch.cat([torch.arange(s.start, s.end, dtype=torch.int64) for s in self.segments])


def zigzag_segments(T: int, world: int, kpool: int) -> List[List[Segment]]:
    """2W blocks of one sequence on pool boundaries; rank r holds blocks r and
    2W-1-r (in that order).  Blocks are ceil(T / 2W) rounded up to a multiple
    of kpool; the last block takes what remains (possibly nothing)."""
    nb = 2 * world
    B = -(-T // nb)
    B = -(-B // kpool) * kpool
    bounds = [min(i * B, T) for i in range(nb)] + [T]
    blocks = [Segment(bounds[i], bounds[i + 1], 0, 0, 0) for i in range(nb)]
    # empty blocks (short sequences) are left out
    return [[b for b in (blocks[r], blocks[nb - 1 - r]) if b.rows > 0] for r in range(world)]


def document_segments(cu_seqlens: Sequence[int], world: int, kpool: int) -> List[List[Segment]]:
    """Contiguous runs of whole documents, cut where the running causal work
    (sum of L_d^2) passes (r+1)/W of the total; a rank may receive none."""
    cu = [int(x) for x in cu_seqlens]
    n = len(cu) - 1
    pools, acc = [], 0
    for d in range(n):
        pools.append(acc)
        acc += (cu[d + 1] - cu[d]) // kpool
    cost = [(cu[d + 1] - cu[d]) ** 2 for d in range(n)]
    total = float(sum(cost)) or 1.0
    out: List[List[Segment]] = [[] for _ in range(world)]
    run, r = 0.0, 0
    for d in range(n):
        # move to the next rank when this document's midpoint lies past its share
        while r < world - 1 and run + cost[d] / 2.0 > (r + 1) * total / world:
            r += 1
        out[r].append(Segment(cu[d], cu[d + 1], d, cu[d], pools[d]))
        run += cost[d]
    return out


def plan_shards(T: int, world: int, rank: int, kpool: int,
                cu_seqlens: Optional[Sequence[int]] = None) -> ShardPlan:
    """The shard plan of `rank`: zigzag for one sequence, whole documents for
    packed documents."""
    if not 0 <= rank < world:
        raise ValueError("rank %d outside world %d" % (rank, world))
    if kpool < 1:
        raise ValueError("kpool must be >= 1")
    if cu_seqlens is None or len(cu_seqlens) <= 2:
        segs = zigzag_segments(T, world, kpool)
        layout = "zigzag"
        P = T // kpool
    else:
        cu = [int(x) for x in cu_seqlens]
        if cu[0] != 0 or cu[-1] != T or any(b < a for a, b in zip(cu[:-1], cu[1:])):
            raise ValueError("cu_seqlens must run from 0 to T, non-decreasing")
        segs = document_segments(cu, world, kpool)
        layout = "documents"
        P = sum((b - a) // kpool for a, b in zip(cu[:-1], cu[1:]))
    return ShardPlan(rank, world, kpool, T, P, layout, tuple(segs[rank]),
                     tuple(tuple(s) for s in segs))


@dataclass
class LocalPools:
    """Pooled keys of one rank's segments, concatenated in segment order:
    pk bf16 [n, D] (BF16 mode) or pk8 E4M3 codes [n, D] + pks fp32 [n]."""
    pk: Optional[torch.Tensor] = None
    pk8: Optional[torch.Tensor] = None
    pks: Optional[torch.Tensor] = None


class DeviceOps:
    """The four operations on the GPU through the C ABI (the product path)."""

    def __init__(self, device):
        from . import binding as B
        self.B = B
        self.device = torch.device(device)

    def tensor(self, values) -> torch.Tensor:
        return torch.tensor(list(values), dtype=torch.int32, device=self.device)

    def compress(self, k, gate, ape, kpool, cu, cu_pools, P, fp8) -> LocalPools:
        n_docs = cu.numel() - 1
        out = self.B.kpool_compress(k, gate, ape, kpool, cu if n_docs > 1 else None,
                                    cu_pools if n_docs > 1 else None, P, fp8=fp8)
        if fp8:
            return LocalPools(pk=out[0], pk8=out[1], pks=out[2])
        return LocalPools(pk=out)

    def quantize(self, q):
        return self.B.kpool_quantize_fp8(q)

    def score_at(self, q, w, pools: LocalPools, kpool, index_topk, cu_q, q_pos, cu_pools,
                 q_scale, out):
        if q_scale is not None:
            return self.B.kpool_score_topk_at(q, w, pools.pk8, kpool, index_topk, cu_q, q_pos,
                                              cu_pools, q_scale=q_scale, pk_scale=pools.pks,
                                              out=out)
        return self.B.kpool_score_topk_at(q, w, pools.pk, kpool, index_topk, cu_q, q_pos,
                                          cu_pools, out=out)

    def expand_at(self, pool_idx, kpool, index_topk, cu_q, q_pos, cu_k, cu_pools, tail, out):
        return self.B.kpool_expand_indices_at(pool_idx, kpool, index_topk, cu_q, q_pos, cu_k,
                                              cu_pools, tail, out=out)


def _empty_like_rows(t: torch.Tensor, rows: int) -> torch.Tensor:
    return torch.empty((rows,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)


class ShardedIndexer:
    """The indexer pass of one rank under a ShardPlan.

    Inputs on each rank are the rows of its segments, concatenated in segment
    order (the context-parallel layout): q [n, H, D] bf16, k and gate [n, D]
    bf16, w [n, H] fp32; ape [kpool, D] fp32 is replicated.  The result is
    tok_idx [n, Kp*kpool + kpool - 1] int32 for the same rows, with global
    token indices, equal row for row to the single-GPU pass on the whole
    input.

    The pass runs in three phases so that a caller can drive them one by one:
    local_pools (compression, and the FP8 cast of q), assemble (after the
    exchange of pooled keys, when the layout needs it) and score_expand."""

    def __init__(self, plan: ShardPlan, index_topk: int, tail: bool = True, fp8: bool = False,
                 ops=None, device="cuda"):
        if index_topk % plan.kpool:
            raise ValueError("index_topk must be a multiple of kpool")
        self.plan = plan
        self.index_topk = index_topk
        self.tail = tail
        self.fp8 = fp8
        self.ops = ops if ops is not None else DeviceOps(device)
        self._index_cache = {}

    def _index(self, values) -> torch.Tensor:
        """An int32 index array on the ops' device, made once per distinct value
        list (the plan's arrays do not change between passes)."""
        key = tuple(int(v) for v in values)
        t = self._index_cache.get(key)
        if t is None:
            t = self._index_cache[key] = self.ops.tensor(key)
        return t

    # ---- phase 1 ------------------------------------------------------------
    def local_pools(self, k, gate, ape) -> LocalPools:
        """Compress the complete pools of this rank's segments (each segment
        starts on a pool boundary of its document, so these are exactly the
        document's pools over the segment)."""
        pl, kp = self.plan, self.plan.kpool
        if k.shape[0] != pl.local_rows:
            raise ValueError("k has %d rows, the plan gives this rank %d"
                             % (k.shape[0], pl.local_rows))
        cu, cp = [0], [0]
        for s in pl.segments:
            cu.append(cu[-1] + s.rows)
            cp.append(cp[-1] + s.pools(kp))
        return self.ops.compress(k, gate, ape, kp, self._index(cu), self._index(cp), cp[-1],
                                 self.fp8)

    # ---- phase 2 --------------------------------------------------------------
    def exchange_parts(self, local: LocalPools) -> List[torch.Tensor]:
        """The tensors this rank sends in the all-gather, padded to the largest
        rank's pool count (every rank knows every rank's count from the plan)."""
        pmax = max(self.plan.local_pools(r) for r in range(self.plan.world))
        parts = [local.pk8, local.pks] if self.fp8 else [local.pk]
        out = []
        for t in parts:
            buf = torch.zeros((pmax,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
            buf[: t.shape[0]].copy_(t)
            out.append(buf)
        return out

    def assemble(self, gathered: Sequence[Sequence[torch.Tensor]]) -> LocalPools:
        """Global pooled keys [P_total, ...] from every rank's exchange_parts
        (gathered[r] = rank r's list): each rank's segments' pools are copied
        to their global pool rows."""
        pl, kp = self.plan, self.plan.kpool
        glob = [torch.empty((pl.P_total,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
                for t in gathered[0]]
        for r in range(pl.world):
            o = 0
            for s in pl.all_segments[r]:
                n = s.pools(kp)
                g0 = s.first_pool(kp)
                for dst, src in zip(glob, gathered[r]):
                    dst[g0:g0 + n].copy_(src[o:o + n])
                o += n
        if self.fp8:
            return LocalPools(pk8=glob[0], pks=glob[1])
        return LocalPools(pk=glob[0])

    # ---- phase 3 --------------------------------------------------------------
    def score_expand(self, q, w, pools: LocalPools, q_scale=None):
        """Pool selection and expansion of this rank's query rows.  `pools` is
        the global pooled keys (zigzag) or the rank's own (documents).
        Returns (tok_idx, pool_idx, pool_score) for the local rows."""
        pl, kp, topk = self.plan, self.plan.kpool, self.index_topk
        Kp = topk // kp
        n = pl.local_rows
        dev = q.device
        pool_idx = torch.empty(n, Kp, dtype=torch.int32, device=dev)
        pool_score = torch.empty(n, Kp, dtype=torch.float32, device=dev)
        tok = torch.empty(n, Kp * kp + kp - 1, dtype=torch.int32, device=dev)
        if n == 0:
            return tok, pool_idx, pool_score
        T = self._index
        if pl.layout == "zigzag":
            # one positioned call per block: the blocks of a rank are two pieces
            # of one sequence and both score the whole sequence's pooled keys
            cp = T([0, pl.P_total])
            ck = T([0, pl.T])
            for s, o in zip(pl.segments, pl.row_offsets()):
                if s.rows == 0:
                    continue
                sl = slice(o, o + s.rows)
                cq, qp = T([0, s.rows]), T([s.start])
                self.ops.score_at(q[sl], w[sl], pools, kp, topk, cq, qp, cp,
                                  q_scale[sl] if q_scale is not None else None,
                                  (pool_idx[sl], pool_score[sl]))
                self.ops.expand_at(pool_idx[sl], kp, topk, cq, qp, ck, cp, self.tail, tok[sl])
        else:
            # the rank's whole documents with their own pooled keys; expansion
            # adds each document's global start
            cu_q, cp, ck = [0], [0], []
            for s in pl.segments:
                cu_q.append(cu_q[-1] + s.rows)
                cp.append(cp[-1] + s.pools(kp))
                ck.append(s.doc_start)
            ck.append(pl.segments[-1].end)
            cq, qp = T(cu_q), T([0] * len(pl.segments))
            cpt = T(cp)
            self.ops.score_at(q, w, pools, kp, topk, cq, qp, cpt, q_scale, (pool_idx, pool_score))
            self.ops.expand_at(pool_idx, kp, topk, cq, qp, T(ck), cpt, self.tail, tok)
        return tok, pool_idx, pool_score

    # ---- the whole pass --------------------------------------------------------
    def forward(self, q, k, gate, ape, w, group=None):
        """The rank's pass with torch.distributed for the exchange (NCCL between
        GPUs).  Returns tok_idx for the local rows."""
        pools = self.local_pools(k, gate, ape)
        if self.plan.exchange:
            import torch.distributed as dist
            parts = self.exchange_parts(pools)
            gathered = [[torch.empty_like(p) for p in parts] for _ in range(self.plan.world)]
            for i, p in enumerate(parts):
                dist.all_gather([g[i] for g in gathered], p, group=group)
            pools = self.assemble(gathered)
        q_scale = None
        if self.fp8:
            q, q_scale = self.ops.quantize(q)
        tok, _, _ = self.score_expand(q, w, pools, q_scale)
        return tok


def shard_rows(x: torch.Tensor, plan: ShardPlan) -> torch.Tensor:
    """This rank's rows of a full [T, ...] tensor, in local order (a helper for
    benchmarks and tests that hold the whole input on every rank)."""
    if not plan.segments:
        return x[:0].contiguous()
    return torch.cat([x[s.start:s.end] for s in plan.segments]).contiguous()
