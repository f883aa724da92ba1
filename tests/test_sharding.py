"""Query-sharded indexer (sparse_attention_kpool_compress_gb300.sharding) on CPU
ranks: the shard plans, and the whole sharded pass on world sizes 2 and 3
over gloo with the CPU oracle standing in for the four device operations.
Every rank holds only its own rows (the context-parallel layout); ranks
exchange pooled keys with the same all-gather the GPU path uses; the rows
reassembled from all ranks must equal the oracle's unsharded pass bit for
bit (zigzag one-sequence layout in BF16 and FP8 mode, whole-document layout
for packed documents)."""
import os
import random
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_attention_kpool_compress_gb300 import sharding as S  # noqa: E402
from sparse_attention_kpool_compress_gb300 import workloads as W  # noqa: E402


# ---------------------------------------------------------------------------
# shard plans
# ---------------------------------------------------------------------------

def _causal_work(plan, cu):
    """Sum over the rank's query rows of their complete causal pools."""
    cu = np.asarray(cu, np.int64)
    tot = 0
    for s in plan.segments:
        t = np.arange(s.start, s.end)
        tau = t - s.doc_start
        tot += int(((tau + 1) // plan.kpool).sum())
    return tot


@pytest.mark.parametrize("T,world,kp", [(131072, 2, 4), (131072, 8, 4), (1000, 3, 4),
                                        (37, 4, 4), (5000, 5, 3), (64, 1, 4)])
def test_zigzag_plan_covers_and_balances(T, world, kp):
    plans = [S.plan_shards(T, world, r, kp) for r in range(world)]
    rows = np.concatenate([p.local_row_index().numpy() for p in plans])
    assert np.array_equal(np.sort(rows), np.arange(T))
    assert sum(p.local_pools() for p in plans) == T // kp == plans[0].P_total
    for p in plans:
        assert p.layout == "zigzag" and p.exchange == (world > 1)
        for s in p.segments:
            assert s.start % kp == 0 and s.doc == 0 and s.pool_base == 0
            assert s.first_pool(kp) == s.start // kp
    if T >= 64 * world * kp:
        # equal shares of the causal triangle, up to the rounding of the blocks
        # to pools (the last block is shorter by at most 2W * kpool rows)
        works = [_causal_work(p, [0, T]) for p in plans]
        assert max(works) <= (1.01 if T >= 16384 else 1.1) * min(works)


def test_document_plan_whole_documents():
    wl = W.Workload("s", T=32768, H=4, D=32, kpool=4, index_topk=64, n_docs=16,
                    doc_len_range=(256, 4096))
    cu = W.make_inputs(wl).cu_seqlens.tolist()
    for world in (1, 2, 3, 4, 16, 20):
        plans = [S.plan_shards(32768, world, r, 4, cu) for r in range(world)]
        docs = [s.doc for p in plans for s in p.segments]
        assert docs == list(range(16))   # every document once, in order, runs contiguous
        for p in plans:
            assert p.layout == "documents" and not p.exchange
            for s in p.segments:
                assert (s.start, s.end) == (cu[s.doc], cu[s.doc + 1])
        if world <= 4:
            works = [sum((s.end - s.start) ** 2 for s in p.segments) for p in plans]
            total = sum(works)
            assert max(works) <= total / world + max((b - a) ** 2 for a, b in zip(cu, cu[1:]))


def test_plan_rejects_bad_input():
    with pytest.raises(ValueError):
        S.plan_shards(100, 2, 2, 4)
    with pytest.raises(ValueError):
        S.plan_shards(100, 2, 0, 4, [0, 60, 50, 100])


# ---------------------------------------------------------------------------
# the sharded pass with the oracle as the device
# ---------------------------------------------------------------------------

class OracleOps:
    """The four operations on CPU through the oracle (test infrastructure):
    torch CPU tensors in and out, the oracle's arithmetic inside."""

    def __init__(self):
        import oracle
        oracle.build()
        self.ora = oracle

    def tensor(self, values):
        return torch.tensor(list(values), dtype=torch.int32)

    def compress(self, k, gate, ape, kpool, cu, cu_pools, P, fp8):
        cs = cu.numpy() if cu.numel() > 2 else None
        pkb = self.ora.compress(W.bits(k), W.bits(gate), ape.numpy(), cs, kpool)
        assert pkb.shape[0] == P
        pk = torch.from_numpy(pkb.view(np.int16).copy()).view(torch.bfloat16)
        if not fp8:
            return S.LocalPools(pk=pk)
        codes, scales = self.ora.fp8_rows(pkb) if P else (np.zeros((0, pkb.shape[1]), np.uint8),
                                                         np.zeros(0, np.float32))
        return S.LocalPools(pk=pk, pk8=torch.from_numpy(codes.copy()),
                            pks=torch.from_numpy(scales.copy()))

    def quantize(self, q):
        T, H, D = q.shape
        codes, scales = self.ora.fp8_rows(W.bits(q).reshape(-1, D))
        return (torch.from_numpy(codes.reshape(T, H, D).copy()),
                torch.from_numpy(scales.reshape(T, H).copy()))

    def score_at(self, q, w, pools, kpool, index_topk, cu_q, q_pos, cu_pools, q_scale, out):
        # the oracle derives each document's pools from its key counts: a
        # document of P_d pools is given P_d * kpool keys
        ck = cu_pools.numpy().astype(np.int64) * kpool
        if q_scale is not None:
            ops = self.ora.Operands(q.numpy(), w.numpy(), pools.pk8.numpy(), q_scale.numpy(),
                                    pools.pks.numpy())
        else:
            ops = self.ora.Operands(W.bits(q), w.numpy(), W.bits(pools.pk))
        rows = np.arange(q.shape[0])
        o = self.ora.select_rows_at(ops, cu_q.numpy(), q_pos.numpy(), ck.astype(np.int32), kpool,
                                    index_topk // kpool, rows)
        out[0].copy_(torch.from_numpy(o["sel"]))
        out[1].copy_(torch.from_numpy(o["sel_score"].astype(np.float32)))
        return out

    def expand_at(self, pool_idx, kpool, index_topk, cu_q, q_pos, cu_k, cu_pools, tail, out):
        rows = np.arange(pool_idx.shape[0])
        tok = self.ora.expand_rows_at(pool_idx.numpy(), cu_q.numpy(), q_pos.numpy(),
                                      cu_k.numpy(), kpool, index_topk // kpool, tail, rows)
        out.copy_(torch.from_numpy(tok))
        return out


def _workload(kind):
    if kind == "zigzag":
        return W.Workload("sz", T=1500, H=4, D=32, kpool=4, index_topk=64)
    if kind == "zigzag_fp8":
        return W.Workload("sz8", T=1000, H=2, D=128, kpool=4, index_topk=48, fp8=True)
    return W.Workload("sd", T=3000, H=4, D=32, kpool=4, index_topk=64, n_docs=7,
                      doc_len_range=(50, 900))


def _unsharded(wl, inp):
    import oracle as ora
    ora.build()
    cu = inp.cu_seqlens.numpy() if inp.cu_seqlens.numel() > 2 else None
    pkb = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(), cu, wl.kpool)
    if wl.fp8:
        pc, ps = ora.fp8_rows(pkb)
        qc, qs = ora.fp8_rows(W.bits(inp.q).reshape(-1, wl.D))
        ops = ora.Operands(qc.reshape(wl.T, wl.H, wl.D), inp.w.numpy(), pc,
                           qs.reshape(wl.T, wl.H), ps)
    else:
        ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    rows = np.arange(wl.T)
    o = ora.select_rows(ops, cu, wl.kpool, wl.Kp, rows)
    return ora.expand_rows(o["sel"], cu, wl.T, wl.kpool, wl.Kp, wl.tail, rows)


def _worker(rank, world, port, kind, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = _workload(kind)
        inp = W.make_inputs(wl, seed=7)
        cu = inp.cu_seqlens.tolist() if inp.cu_seqlens.numel() > 2 else None
        plan = S.plan_shards(wl.T, world, rank, wl.kpool, cu)
        # this rank holds only its own rows
        q, k, gate, w = (S.shard_rows(x, plan) for x in (inp.q, inp.k, inp.gate, inp.w))
        idx = S.ShardedIndexer(plan, wl.index_topk, wl.tail, wl.fp8, ops=OracleOps())
        pools = idx.local_pools(k, gate, inp.ape)
        if plan.exchange:
            # gloo moves the parts as raw bytes (it has no bf16)
            parts = idx.exchange_parts(pools)
            dts = [p.dtype for p in parts]
            raw = [p.view(torch.uint8) for p in parts]
            gathered = [[torch.empty_like(p) for p in raw] for _ in range(world)]
            for i, p in enumerate(raw):
                dist.all_gather([g[i] for g in gathered], p)
            gathered = [[g.view(dt) for g, dt in zip(gr, dts)] for gr in gathered]
            pools = idx.assemble(gathered)
        q_scale = None
        if wl.fp8:
            q, q_scale = idx.ops.quantize(q)
        tok, _, _ = idx.score_expand(q, w, pools, q_scale)
        res = [None] * world
        dist.all_gather_object(res, (plan.local_row_index().numpy(), tok.numpy()))
        if rank == 0:
            full = np.full((wl.T, tok.shape[1]), -7, np.int32)
            for rows, t in res:
                full[rows] = t
            out.put(("ok", kind, world, full, plan.layout))
    except Exception as e:   # report to the parent instead of hanging it
        out.put(("error", repr(e)))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("kind,world", [("zigzag", 2), ("zigzag", 3), ("zigzag_fp8", 2),
                                        ("documents", 2), ("documents", 3)])
def test_sharded_pass_equals_unsharded_oracle(kind, world):
    port = 29500 + random.randint(0, 4000)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, kind, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
    assert res[0] == "ok", res
    for p in procs:
        assert p.exitcode == 0
    _, _, _, full, layout = res
    assert layout == ("documents" if kind == "documents" else "zigzag")
    wl = _workload(kind)
    want = _unsharded(wl, W.make_inputs(wl, seed=7))
    assert np.array_equal(full, want)
