"""Positioned queries (decode and chunked prefill): kpool_score_topk_at and
kpool_expand_indices_at against the oracle's select_rows_at / expand_rows_at,
and against the rows of a full prefill computed by the GPU itself."""
import numpy as np
import pytest
import torch

from sparse_attention_kpool_compress_gb300 import workloads as W
from kpool_checks import check_selection

pytestmark = pytest.mark.gpu

TOL = 1e-3


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_kpool_compress_gb300 as K
    return K


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _keys(seed=3):
    wl = W.Workload("kv", T=6000, H=64, D=128, kpool=4, index_topk=512, n_docs=3,
                    doc_len_range=(1000, 3000))
    inp = W.make_inputs(wl, seed=seed)
    return wl, inp, inp.cu_seqlens.numpy()


def _run(K, ora, wl, inp, cu_k, chunks):
    """chunks: per document (a, b) document-local query positions [a, b)."""
    dev = torch.device("cuda")
    kp, Kp = wl.kpool, wl.Kp
    pkb = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(), cu_k, kp)
    cu_pools_h, P = K.kpool_num_pools(torch.from_numpy(cu_k), wl.T, kp)
    rows = np.concatenate([np.arange(cu_k[d] + a, cu_k[d] + b) for d, (a, b) in enumerate(chunks)])
    cq = np.concatenate([[0], np.cumsum([b - a for a, b in chunks])]).astype(np.int32)
    qpos = np.array([a for a, _ in chunks], np.int32)
    q = inp.q[torch.from_numpy(rows)].contiguous()
    w = inp.w[torch.from_numpy(rows)].contiguous()
    d_cq, d_qpos = torch.from_numpy(cq).to(dev), torch.from_numpy(qpos).to(dev)
    d_cp, d_ck = cu_pools_h.to(dev), torch.from_numpy(cu_k).to(dev)
    idx, sc = K.kpool_score_topk_at(q.to(dev), w.to(dev), _bf16(pkb).to(dev), kp, wl.index_topk,
                                    d_cq, d_qpos, d_cp)
    tok = K.kpool_expand_indices_at(idx, kp, wl.index_topk, d_cq, d_qpos, d_ck, d_cp, True)
    torch.cuda.synchronize()
    ops = ora.Operands(W.bits(q), w.numpy(), pkb)
    return rows, cq, qpos, pkb, ops, idx.cpu().numpy(), sc.cpu().numpy(), tok.cpu().numpy()


def _check_vs_oracle(ora, ops, cq, qpos, cu_k, wl, idx, sc, tok):
    n = idx.shape[0]
    o = ora.select_rows_at(ops, cq, qpos, cu_k, wl.kpool, wl.Kp, np.arange(n))
    # reuse the generic checker through a small adapter over the _at oracle
    class At:
        select_rows = staticmethod(lambda ops_, cu, kp, Kp, rows: ora.select_rows_at(
            ops_, cq, qpos, cu_k, kp, Kp, rows))
        score_pairs = staticmethod(lambda ops_, cu, kp, rows, pools: ora.score_pairs_at(
            ops_, cq, qpos, cu_k, kp, rows, pools))
    st = check_selection(At, ops, None, wl.kpool, wl.Kp, np.arange(n), idx, sc, TOL, "at")
    want = ora.expand_rows_at(idx, cq, qpos, cu_k, wl.kpool, wl.Kp, True, np.arange(n))
    assert np.array_equal(tok, want)
    return o, st


def test_chunked_prefill(K, ora):
    wl, inp, cu_k = _keys()
    L = np.diff(cu_k)
    chunks = [(int(L[d] // 3), int(2 * L[d] // 3)) for d in range(3)]
    rows, cq, qpos, pkb, ops, idx, sc, tok = _run(K, ora, wl, inp, cu_k, chunks)
    _check_vs_oracle(ora, ops, cq, qpos, cu_k, wl, idx, sc, tok)
    # the same rows of a GPU full prefill are identical, bit for bit
    dev = torch.device("cuda")
    cu_pools_h, _ = K.kpool_num_pools(torch.from_numpy(cu_k), wl.T, wl.kpool)
    fidx, fsc = K.kpool_score_topk(inp.q.to(dev), inp.w.to(dev), _bf16(pkb).to(dev), wl.kpool,
                                   wl.index_topk, torch.from_numpy(cu_k).to(dev),
                                   cu_pools_h.to(dev))
    ftok = K.kpool_expand_indices(fidx, wl.kpool, wl.index_topk, True,
                                  torch.from_numpy(cu_k).to(dev), cu_pools_h.to(dev))
    torch.cuda.synchronize()
    assert np.array_equal(fidx.cpu().numpy()[rows], idx)
    assert np.array_equal(fsc.cpu().numpy()[rows], sc)
    assert np.array_equal(ftok.cpu().numpy()[rows], tok)


def test_decode_one_query_per_document(K, ora):
    wl, inp, cu_k = _keys(seed=4)
    L = np.diff(cu_k)
    chunks = [(int(L[d] - 1), int(L[d])) for d in range(3)]
    rows, cq, qpos, pkb, ops, idx, sc, tok = _run(K, ora, wl, inp, cu_k, chunks)
    o, _ = _check_vs_oracle(ora, ops, cq, qpos, cu_k, wl, idx, sc, tok)
    assert np.all(o["n_sel"] == np.minimum(L // wl.kpool, wl.Kp))


def test_positioned_small_ragged(K, ora):
    """Tiny documents, chunks at the start, the middle and a ragged tail."""
    wl = W.Workload("kv2", T=700, H=16, D=64, kpool=4, index_topk=40, n_docs=4,
                    doc_len_range=(30, 400))
    inp = W.make_inputs(wl, seed=9)
    cu_k = inp.cu_seqlens.numpy()
    L = np.diff(cu_k)
    chunks = [(0, int(min(L[0], 5))), (int(L[1] // 2), int(L[1])), (1, 2), (int(L[3] - 7), int(L[3]))]
    rows, cq, qpos, pkb, ops, idx, sc, tok = _run(K, ora, wl, inp, cu_k, chunks)
    _check_vs_oracle(ora, ops, cq, qpos, cu_k, wl, idx, sc, tok)


def _fullsize(K, ora, name, n_sample):
    """The positioned workload at full size in the benchmark's launch
    configuration: pooled keys (GPU vs oracle), the scorer on the oracle's
    pooled keys for sampled query rows, and bit-exact expansion."""
    from kpool_checks import bf16_bits, check_pooled_keys
    dev = torch.device("cuda")
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    cu_k = inp.cu_seqlens.numpy()
    multi = len(cu_k) > 2
    cu_pools_h, P = K.kpool_num_pools(inp.cu_seqlens, wl.T, wl.kpool)
    d_ck, d_cp = inp.cu_seqlens.to(dev), cu_pools_h.to(dev)
    pk = K.kpool_compress(inp.k.to(dev), inp.gate.to(dev), inp.ape.to(dev), wl.kpool,
                          d_ck if multi else None, d_cp if multi else None, P)
    pkb, exact, cond = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(),
                                    cu_k if multi else None, wl.kpool, want_exact=True,
                                    want_cond=True)
    check_pooled_keys(bf16_bits(pk), pkb, exact, cond, name)
    cq, qp = inp.cu_q.numpy(), inp.q_pos.numpy()
    d_cq, d_qp = inp.cu_q.to(dev), inp.q_pos.to(dev)
    q, w = inp.q.to(dev), inp.w.to(dev)
    idx, sc = K.kpool_score_topk_at(q, w, _bf16(pkb).to(dev), wl.kpool, wl.index_topk, d_cq, d_qp,
                                    d_cp)
    tok = K.kpool_expand_indices_at(idx, wl.kpool, wl.index_topk, d_cq, d_qp, d_ck, d_cp, True)
    torch.cuda.synchronize()
    rows = W.sample_rows(inp.Tq, n_sample).numpy()
    idx_h, sc_h, tok_h = idx.cpu().numpy(), sc.cpu().numpy(), tok.cpu().numpy()
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)

    class At:
        select_rows = staticmethod(lambda ops_, cu, kp, Kp, r: ora.select_rows_at(
            ops_, cq, qp, cu_k, kp, Kp, r))
        score_pairs = staticmethod(lambda ops_, cu, kp, r, p: ora.score_pairs_at(
            ops_, cq, qp, cu_k, kp, r, p))
    check_selection(At, ops, None, wl.kpool, wl.Kp, rows, idx_h[rows], sc_h[rows], TOL, name)
    want = ora.expand_rows_at(idx_h[rows], cq, qp, cu_k, wl.kpool, wl.Kp, True, rows)
    assert np.array_equal(tok_h[rows], want)
    return inp, idx_h


@pytest.mark.slow
def test_fullsize_chunk_16k_of_128k(K, ora):
    inp, idx = _fullsize(K, ora, "chunk_16k_of_128k", 512)
    # every chunk query sees more complete pools than the budget
    assert np.all(idx >= 0)


@pytest.mark.slow
def test_fullsize_decode_128x32k(K, ora):
    inp, idx = _fullsize(K, ora, "decode_128x32k", 1024)   # 128 rows: all of them
    assert inp.Tq == 128 and np.all(idx >= 0)


def _split_vs_unsplit(K, ora, wl, n_check, expect_split=True):
    """kpool_score_topk_at with a workspace that enables the split-pool
    schedule against the same call with the minimal workspace (one unit per
    query tile): identical outputs, bit for bit; plus oracle rows (in FP8 mode
    on the GPU's own E4M3 codes and scales)."""
    dev = torch.device("cuda")
    inp = W.make_inputs(wl)
    cu_k = inp.cu_seqlens.numpy()
    n_docs = len(cu_k) - 1
    cu_pools_h, P = K.kpool_num_pools(inp.cu_seqlens, wl.T, wl.kpool)
    d_ck, d_cp = inp.cu_seqlens.to(dev), cu_pools_h.to(dev)
    d_cq, d_qp = inp.cu_q.to(dev), inp.q_pos.to(dev)
    q, w = inp.q.to(dev), inp.w.to(dev)
    qs = pks = None
    if wl.fp8:
        pk_bf, pk, pks = K.kpool_compress(inp.k.to(dev), inp.gate.to(dev), inp.ape.to(dev),
                                          wl.kpool, d_ck, d_cp, P, fp8=True)
        q, qs = K.kpool_quantize_fp8(q)
    else:
        pk = K.kpool_compress(inp.k.to(dev), inp.gate.to(dev), inp.ape.to(dev), wl.kpool, d_ck,
                              d_cp, P)
    Tq, H = inp.Tq, wl.H
    ws_split = K.new_workspace(Tq, H, n_docs, dev, wl.kpool, wl.index_topk)
    ws_one = K.new_workspace(Tq, H, n_docs, dev)
    assert ws_split.numel() > ws_one.numel()
    a = K.kpool_score_topk_at(q, w, pk, wl.kpool, wl.index_topk, d_cq, d_qp, d_cp, q_scale=qs,
                              pk_scale=pks, workspace=ws_split)
    b = K.kpool_score_topk_at(q, w, pk, wl.kpool, wl.index_topk, d_cq, d_qp, d_cp, q_scale=qs,
                              pk_scale=pks, workspace=ws_one)
    torch.cuda.synchronize()
    assert K.kpool_read_status(ws_split) == 0 and K.kpool_read_status(ws_one) == 0
    # the workspace header's third word is the number of scheduled units: more
    # units than query tiles means some tile's pools were split
    qt = 256 // H
    tiles = int(sum((int(n) + qt - 1) // qt for n in np.diff(inp.cu_q.numpy())))
    units = int(ws_split[:12].view(torch.int32)[2])
    assert (units > tiles) == expect_split, (units, tiles)
    assert torch.equal(a[0], b[0])
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
    cq, qp = inp.cu_q.numpy(), inp.q_pos.numpy()
    rows = np.unique(np.linspace(0, Tq - 1, n_check).astype(np.int64))
    if wl.fp8:
        ops = ora.Operands(q.cpu().numpy(), inp.w.numpy(), pk.cpu().numpy(), qs.cpu().numpy(),
                           pks.cpu().numpy())
    else:
        from kpool_checks import bf16_bits
        ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), bf16_bits(pk))

    class At:
        select_rows = staticmethod(lambda ops_, cu, kp, Kp, r: ora.select_rows_at(
            ops_, cq, qp, cu_k, kp, Kp, r))
        score_pairs = staticmethod(lambda ops_, cu, kp, r, p: ora.score_pairs_at(
            ops_, cq, qp, cu_k, kp, r, p))
    idx, sc = a[0].cpu().numpy(), a[1].cpu().numpy()
    check_selection(At, ops, None, wl.kpool, wl.Kp, rows, idx[rows], sc[rows], TOL, wl.name)
    return idx


def test_split_schedule_decode_long_documents(K, ora):
    """48 decode queries over documents of 2K-30K keys: pool lists of up to 60
    tiles, cut into up to 16 units each."""
    wl = W.Workload("split_decode", T=48 * 16384, H=64, D=128, kpool=4, index_topk=2048,
                    n_docs=48, doc_len_range=(2048, 30720), queries="last", seed=21)
    idx = _split_vs_unsplit(K, ora, wl, 12)
    assert np.all(idx >= 0)


def test_split_schedule_chunks_share_units(K, ora):
    """Chunks of 37 queries (full and ragged query tiles) at the end of two
    long documents: every query of a split tile is merged."""
    wl = W.Workload("split_chunk", T=2 * 20000, H=64, D=128, kpool=4, index_topk=512,
                    n_docs=2, equal_docs=True, queries="chunk:37", seed=22)
    _split_vs_unsplit(K, ora, wl, 16)


def test_split_schedule_small_heads_and_large_budget(K, ora):
    """H = 16 (16 queries per tile) with Kp = 256; kpool = 2 with Kp = 768 (split,
    larger partial lists); kpool = 2 with Kp = 1024, more than half a query's
    candidate capacity in the split layout, so the lists cannot be merged in
    place and the call runs unsplit."""
    wl = W.Workload("split_h16", T=8 * 24000, H=16, D=64, kpool=4, index_topk=1024,
                    n_docs=8, equal_docs=True, queries="chunk:21", seed=23)
    _split_vs_unsplit(K, ora, wl, 16)
    wl = W.Workload("split_kp2", T=4 * 12000, H=64, D=128, kpool=2, index_topk=1536,
                    n_docs=4, equal_docs=True, queries="last", seed=24)
    _split_vs_unsplit(K, ora, wl, 4)
    wl = W.Workload("split_kp2_big", T=4 * 12000, H=64, D=128, kpool=2, index_topk=2048,
                    n_docs=4, equal_docs=True, queries="last", seed=27)
    _split_vs_unsplit(K, ora, wl, 4, expect_split=False)


def test_split_schedule_decode_fp8(K, ora):
    """Lone-query tiles in FP8 mode: the per-pool E4M3 scale in the packed
    accumulator loop."""
    wl = W.Workload("split_decode_fp8", T=24 * 16384, H=64, D=128, kpool=4, index_topk=2048,
                    n_docs=24, doc_len_range=(4096, 28672), queries="last", fp8=True, seed=25)
    idx = _split_vs_unsplit(K, ora, wl, 8)
    assert np.all(idx >= 0)


def test_split_schedule_decode_h128(K, ora):
    """H = 128: two pool tiles per accumulator, each query's heads in two
    64-column halves."""
    wl = W.Workload("split_decode_h128", T=16 * 12000, H=128, D=64, kpool=4, index_topk=1024,
                    n_docs=16, doc_len_range=(3000, 20000), queries="last", seed=26)
    _split_vs_unsplit(K, ora, wl, 8)
