"""The query-sharded indexer's device path on one GPU: W ranks emulated one
after another (each runs its own compression, the exchange is a copy of
every rank's pooled keys, then each scores and expands its own rows), so no
kernel ever waits on another rank.  The rows reassembled from the emulated
ranks must equal the single-GPU pass kpool_indexer_forward bit for bit:
zigzag blocks of one sequence (BF16 and FP8) and whole packed documents."""
import numpy as np
import pytest
import torch

from sparse_attention_kpool_compress_gb300 import sharding as S
from sparse_attention_kpool_compress_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_kpool_compress_gb300 as K
    return K


def _emulate(wl, inp, world):
    dev = torch.device("cuda")
    cu = inp.cu_seqlens.tolist() if inp.cu_seqlens.numel() > 2 else None
    plans = [S.plan_shards(wl.T, world, r, wl.kpool, cu) for r in range(world)]
    ranks = []
    for p in plans:
        x = {n: S.shard_rows(getattr(inp, n), p).to(dev) for n in ("q", "k", "gate", "w")}
        idx = S.ShardedIndexer(p, wl.index_topk, wl.tail, wl.fp8, device=dev)
        ranks.append((p, idx, x, idx.local_pools(x["k"], x["gate"], inp.ape.to(dev))))
    # the exchange: every rank receives every rank's padded parts
    gathered = [idx.exchange_parts(pools) for _, idx, _, pools in ranks]
    full = None
    for p, idx, x, pools in ranks:
        use = idx.assemble(gathered) if p.exchange else pools
        q, qs = x["q"], None
        if wl.fp8:
            q, qs = idx.ops.quantize(q)
        tok, _, _ = idx.score_expand(q, x["w"], use, qs)
        torch.cuda.synchronize()
        if full is None:
            full = torch.full((wl.T, tok.shape[1]), -7, dtype=torch.int32)
        full[p.local_row_index()] = tok.cpu()
    return full, plans[0].layout


def _single_gpu(K, wl, inp):
    dev = torch.device("cuda")
    cu_d = cp_d = P = None
    if inp.cu_seqlens.numel() > 2:
        cp_h, P = K.kpool_num_pools(inp.cu_seqlens, wl.T, wl.kpool)
        cu_d, cp_d = inp.cu_seqlens.to(dev), cp_h.to(dev)
    tok, _, _ = K.kpool_indexer_forward(inp.q.to(dev), inp.k.to(dev), inp.gate.to(dev),
                                        inp.ape.to(dev), inp.w.to(dev), wl.kpool, wl.index_topk,
                                        wl.tail, cu_d, cp_d, P, fp8=wl.fp8)
    torch.cuda.synchronize()
    return tok.cpu()


@pytest.mark.parametrize("kind,world", [("zigzag", 2), ("zigzag", 4), ("zigzag_fp8", 3),
                                        ("documents", 3)])
def test_sharded_equals_single_gpu(K, kind, world):
    if kind == "zigzag":
        wl = W.Workload("gz", T=20000, H=64, D=128, kpool=4, index_topk=1024)
    elif kind == "zigzag_fp8":
        wl = W.Workload("gz8", T=12000, H=64, D=128, kpool=4, index_topk=512, fp8=True)
    else:
        wl = W.Workload("gd", T=32768, H=64, D=128, kpool=4, index_topk=2048, n_docs=16,
                        doc_len_range=(256, 4096))
    inp = W.make_inputs(wl, seed=71)
    full, layout = _emulate(wl, inp, world)
    assert layout == ("documents" if kind == "documents" else "zigzag")
    assert torch.equal(full, _single_gpu(K, wl, inp))
