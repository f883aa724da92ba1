"""kpool_score_topk_noalloc: the scoring entry point for callers that cannot
allocate device memory (for example a framework plugin hook that only hands
out its input and output buffers, or a runtime that reserves all device
memory up front).  It keeps its scratch in a fixed array inside the library
instead of a caller workspace.  Checked here, through the C ABI, against the
workspace entry point kpool_score_topk on two calls in a row (the second on
smaller inputs, so a stale schedule from the first call would show), plus
the host-side rejection of sizes beyond its fixed capacity.

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_kpool_compress_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-3


def _inputs(T, H, D, kp, seed):
    wl = W.Workload("noalloc", T=T, H=H, D=D, kpool=kp, index_topk=kp * 64)
    inp = W.make_inputs(wl, seed=seed)
    pk = torch.randn(T // kp, D, generator=torch.Generator().manual_seed(seed + 1))
    return inp, pk.to(torch.bfloat16)


def _run_both(B, inp, pk_cpu, kp, topk):
    dev = torch.device("cuda")
    q, w, pk = inp.q.to(dev), inp.w.to(dev), pk_cpu.to(dev)
    T, H, D = q.shape
    P = pk.shape[0]
    Kp = topk // kp
    L = B._lib
    stream = B._stream(dev)
    idx_a = torch.full((T, Kp), 7, dtype=torch.int32, device=dev)
    sc_a = torch.full((T, Kp), 7.0, dtype=torch.float32, device=dev)
    rc = L.kpool_score_topk_noalloc(B._ptr(q), None, B._ptr(w), B._ptr(pk), None, None, None, 1,
                                    T, P, H, D, kp, topk, 0, B._ptr(idx_a), B._ptr(sc_a), stream)
    assert rc == 0, L.kpool_last_error()
    ws = torch.empty(L.kpool_score_topk_workspace_size(T, H, 1), dtype=torch.uint8, device=dev)
    idx_b = torch.empty_like(idx_a)
    sc_b = torch.empty_like(sc_a)
    rc = L.kpool_score_topk(B._ptr(q), None, B._ptr(w), B._ptr(pk), None, None, None, 1, T, P, H,
                            D, kp, topk, 0, B._ptr(idx_b), B._ptr(sc_b), B._ptr(ws), ws.numel(),
                            stream)
    assert rc == 0, L.kpool_last_error()
    torch.cuda.synchronize()
    assert B.kpool_read_status(ws) == 0
    return (idx_a.cpu().numpy(), sc_a.cpu().numpy()), (idx_b.cpu().numpy(), sc_b.cpu().numpy())


def test_noalloc_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_kpool_compress_gb300 import binding as B
    for T, H, D, kp, seed in [(6000, 64, 128, 4, 31), (1500, 32, 64, 2, 32)]:
        topk = kp * 64
        inp, pk = _inputs(T, H, D, kp, seed)
        (ia, sa), (ib, sb) = _run_both(B, inp, pk, kp, topk)
        assert np.array_equal(ia, ib)
        fin = np.isfinite(sb)
        assert np.array_equal(np.isfinite(sa), fin)
        assert np.all(np.abs(sa[fin] - sb[fin]) <= TOL * np.abs(sb[fin]) + 1e-30)
        for t in (0, kp - 1, T // 2, T - 1):
            n = min((t + 1) // kp, 64)
            assert np.all(ia[t, :n] >= 0) and np.all(ia[t, n:] == -1)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_kpool_compress_gb300 import binding as B
    L = B._lib
    buf = torch.empty(256, dtype=torch.uint8, device="cuda")
    p = B._ptr(buf)
    T = 4 * 131072   # 131072 tiles of 4 queries at H=64, plus one per document
    rc = L.kpool_score_topk_noalloc(p, None, p, p, None, None, None, 1, T, T // 4, 64, 128, 4,
                                    2048, 0, p, p, B._stream(buf.device))
    assert rc == -2
    assert b"131072" in L.kpool_last_error()


def test_noalloc_packed_fp8_through_binding():
    """Packed documents in FP8 mode, through the Python binding: the
    allocation-free call equals kpool_score_topk bit for bit on two calls in a
    row (the documents enter its tile-capacity bound), and its status word
    reads clean."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_kpool_compress_gb300 as K
    dev = torch.device("cuda")
    for seed, T, n_docs in ((61, 9000, 5), (62, 3000, 3)):
        wl = W.Workload("na8", T=T, H=64, D=128, kpool=4, index_topk=512, n_docs=n_docs,
                        doc_len_range=(300, 4000), fp8=True)
        inp = W.make_inputs(wl, seed=seed)
        cu_h, P = K.kpool_num_pools(inp.cu_seqlens, T, 4)
        cu, cp = inp.cu_seqlens.to(dev), cu_h.to(dev)
        _, pk8, pks = K.kpool_compress(inp.k.to(dev), inp.gate.to(dev), inp.ape.to(dev), 4, cu,
                                       cp, P, fp8=True)
        q8, qs = K.kpool_quantize_fp8(inp.q.to(dev))
        w = inp.w.to(dev)
        ia, sa = K.kpool_score_topk_noalloc(q8, w, pk8, 4, 512, cu, cp, q_scale=qs, pk_scale=pks)
        torch.cuda.synchronize()
        assert K.kpool_score_topk_noalloc_status() == 0
        ws = K.new_workspace(T, 64, n_docs, dev)
        ib, sb = K.kpool_score_topk(q8, w, pk8, 4, 512, cu, cp, q_scale=qs, pk_scale=pks,
                                    workspace=ws)
        torch.cuda.synchronize()
        assert K.kpool_read_status(ws) == 0
        assert torch.equal(ia, ib) and torch.equal(sa, sb)


def test_noalloc_status_reports_bad_seqlens():
    """Malformed device cu_seqlens: the allocation-free call writes nothing and
    its status word says so; the next valid call reads clean again."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_kpool_compress_gb300 as K
    T, H, D = 256, 64, 128
    q = torch.randn(T, H, D, device="cuda").to(torch.bfloat16)
    w = torch.randn(T, H, device="cuda")
    pk = torch.randn(T // 4, D, device="cuda").to(torch.bfloat16)
    cu = torch.tensor([0, 200, 100], dtype=torch.int32, device="cuda")   # decreasing, last != T
    cp = torch.tensor([0, 50, 25], dtype=torch.int32, device="cuda")
    K.kpool_score_topk_noalloc(q, w, pk, 4, 32, cu, cp)
    assert K.kpool_score_topk_noalloc_status() & K.STATUS_BAD_SEQLENS
    K.kpool_score_topk_noalloc(q, w, pk, 4, 32)
    assert K.kpool_score_topk_noalloc_status() == 0


def test_noalloc_rejects_tile_overflow_from_documents():
    """T alone fits the fixed scratch (131071 tiles of 4 queries at H = 64) but
    T plus one tile per document does not: rejected on the host, before
    anything is enqueued."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_kpool_compress_gb300 import binding as B
    L = B._lib
    buf = torch.empty(256, dtype=torch.uint8, device="cuda")
    p = B._ptr(buf)
    T = 4 * 131072 - 4 * 8
    cu = torch.zeros(11, dtype=torch.int32, device="cuda")
    rc = L.kpool_score_topk_noalloc(p, None, p, p, None, B._ptr(cu), B._ptr(cu), 10, T, T // 4,
                                    64, 128, 4, 2048, 0, p, p, B._stream(buf.device))
    assert rc == -2
    assert b"131072" in L.kpool_last_error()
