"""The sparse attention over the selection (kpool_sparse_mla_fwd, _pools,
_pools_at) against the oracle's sparse_attn on the same seeded inputs.

Tolerance, from the kernel's arithmetic: scores are exact BF16 products summed
in FP32; the softmax weights p_j are rounded to BF16 (relative error <= 2^-9)
before they multiply kv, while the normaliser sums the FP32 weights; the
output is rounded to BF16 once.  So per element

    |o_gpu - o| <= 2^-9 * sum_j w_j |kv[j, d]| + 2^-9 |o| + (FP32 terms)

with w the exact softmax weights; the tests allow twice that.  lse sums FP32
weights (hardware 2^x, relative error ~2^-22) over at most a few thousand
tokens: 2e-4 absolute.  Paths that list the same tokens in the same order
(fused expansion vs. an explicit token table) run the same arithmetic and are
compared bit for bit."""
import math
import os

import numpy as np
import pytest
import torch

from sparse_attention_kpool_compress_gb300 import workloads as W

pytestmark = pytest.mark.gpu

H, DC = W.MLA_HEADS, W.MLA_DC


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_kpool_compress_gb300 as K
    return K


def _bits(t):
    return W.bits(t.cpu())


def check_attn(ora, q, kv, tok, rows, scale, o_gpu, lse_gpu, name=""):
    """Rows `rows` of the GPU output against the oracle (tok: the rows' token
    lists [len(rows), W])."""
    qb, kvb = _bits(q), _bits(kv)
    o_ref, lse_ref = ora.sparse_attn(qb, kvb, tok, scale, rows)
    kvd = kv.double().numpy()
    qd = q.double().numpy()
    og = o_gpu.float().numpy().astype(np.float64)
    lg = lse_gpu.numpy().astype(np.float64)
    for i, t in enumerate(rows):
        J = tok[i][tok[i] >= 0]
        if len(J) == 0:
            assert np.all(og[i] == 0), (name, t)
            assert np.all(np.isneginf(lg[i])), (name, t)
            continue
        s = scale * (qd[t] @ kvd[J].T)                      # [H, n]
        w = np.exp(s - lse_ref[i][:, None])
        A = w @ np.abs(kvd[J])                              # [H, DC]
        tol = 2.0 ** -8 * (A + np.abs(o_ref[i])) + 1e-7
        err = np.abs(og[i] - o_ref[i])
        bad = err > tol
        assert not bad.any(), (name, int(t), np.argwhere(bad)[:4], err[bad][:4], tol[bad][:4])
        assert np.allclose(lg[i], lse_ref[i], rtol=1e-6, atol=2e-4), (name, int(t))


def _run_tok(K, q, kv, tok, scale):
    dev = torch.device("cuda")
    o, lse = K.kpool_sparse_mla_fwd(q.to(dev), kv.to(dev), torch.from_numpy(tok).to(dev), scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def test_hand_worked(K):
    """tests/golden/sparse_attn_worked.txt through the kernel (all 64 heads
    the same case, latent dims 2.. zero)."""
    from test_oracle_pins import sparse_attn_worked, sparse_attn_worked_inputs
    table, cases = sparse_attn_worked()
    for scale, q0, idx, o0, o1, lse in cases:
        q, kv, tok = sparse_attn_worked_inputs(q0, idx, table, H=H, Dc=DC)
        o, l = _run_tok(K, q, kv, tok, scale)
        o = o.float().numpy()
        assert np.all(o[0, :, 2:] == 0)
        cmax = np.abs(kv.float().numpy()[:, :2]).max(axis=0)
        for d, want in ((0, o0), (1, o1)):
            tol = 2.0 ** -8 * (cmax[d] + abs(want)) + 1e-7
            assert np.all(np.abs(o[0, :, d] - want) <= tol), (idx, d, o[0, :4, d], want)
        if math.isinf(lse):
            assert np.all(np.isneginf(l.numpy()))
        else:
            assert np.allclose(l.numpy(), lse, rtol=1e-6, atol=2e-5), (idx, l[0, :4], lse)


def _random_lists(rng, T, Tk, Wd, sizes, holes=True):
    tok = np.full((T, Wd), -1, np.int32)
    for t in range(T):
        n = sizes[t % len(sizes)]
        if n == 0:
            continue
        v = rng.integers(0, Tk, size=n).astype(np.int32)   # repeats allowed
        if holes and n < Wd:
            pos = np.sort(rng.choice(Wd, size=n, replace=False))
            tok[t, pos] = v
        else:
            tok[t, :n] = v
    return tok


@pytest.mark.parametrize("scale", [W.MLA_SCALE, 0.3])
def test_token_lists_vs_oracle(K, ora, scale):
    """Explicit token lists: empty rows, one token, block edges (127, 128,
    129), several blocks with a ragged last one, -1 holes anywhere and
    repeated indices.  scale 0.3 gives peaked softmaxes whose block maxima
    rise past the reference maximum (the rescale path)."""
    T, Tk, Wd = 96, 3000, 700
    mi = W.make_mla_inputs(T, Tk, seed=5)
    rng = np.random.default_rng(11)
    tok = _random_lists(rng, T, Tk, Wd, [0, 1, 5, 127, 128, 129, 300, 700, 455])
    o, lse = _run_tok(K, mi.q, mi.kv, tok, scale)
    rows = np.arange(T)
    check_attn(ora, mi.q, mi.kv, tok, rows, scale, o, lse, "tok")


def test_rising_scores_rescale_every_block(K, ora):
    """Scores that rise by > 5.5 (8 in base 2) from one block of 128 tokens to
    the next: the reference maximum and the output accumulator are rescaled at
    every block."""
    T, Tk = 4, 1024
    q = torch.zeros(T, H, DC)
    q[:, :, 0] = 1.0
    q[:, :, 1] = torch.linspace(-1, 1, H)
    kv = torch.randn(Tk, DC, generator=torch.Generator().manual_seed(3)) * 0.1
    kv[:, 0] = torch.arange(Tk) * 0.05                    # +6.4 per block of 128
    q, kv = q.to(torch.bfloat16), kv.to(torch.bfloat16)
    tok = np.stack([np.arange(Tk, dtype=np.int32), np.arange(Tk, dtype=np.int32)[::-1].copy(),
                    np.arange(0, Tk, 2, dtype=np.int32).repeat(2), np.full(Tk, 7, np.int32)])
    o, lse = _run_tok(K, q, kv, tok, 1.0)
    check_attn(ora, q, kv, tok, np.arange(T), 1.0, o, lse, "rising")


def _synth_pools(rng, cu, kp, Kp, q_rows=None):
    """Random selections: for each query row (document d, position tau) up to
    Kp distinct complete causal pools, ascending, -1 padded."""
    T = int(cu[-1])
    cu_pools = np.zeros(len(cu), np.int32)
    for d in range(len(cu) - 1):
        cu_pools[d + 1] = cu_pools[d] + (cu[d + 1] - cu[d]) // kp
    sel = np.full((T, Kp), -1, np.int32)
    for d in range(len(cu) - 1):
        for tau in range(cu[d + 1] - cu[d]):
            nc = min((tau + 1) // kp, cu_pools[d + 1] - cu_pools[d])
            n = min(nc, Kp)
            if n:
                sel[cu[d] + tau, :n] = np.sort(rng.choice(nc, size=n, replace=False)) + cu_pools[d]
    return sel, cu_pools


@pytest.mark.parametrize("kp,tail,docs", [(4, True, None), (4, False, None), (3, True, None),
                                          (1, True, None), (8, True, None),
                                          (4, True, (5, (100, 450), None)),
                                          (8, False, (4, (100, 900), 1))])
def test_fused_expansion(K, ora, kp, tail, docs):
    """kpool_sparse_mla_fwd_pools equals kpool_sparse_mla_fwd on the tokens
    kpool_expand_indices writes (bit for bit), and the oracle on the oracle's
    expansion: kpool 1, 3, 4, 8, with and without the tail, one sequence or
    packed documents (one of them empty)."""
    dev = torch.device("cuda")
    T, index_topk = 2500, 96 * kp
    Kp = index_topk // kp
    if docs:
        lens = np.random.default_rng(docs[0]).integers(docs[1][0], docs[1][1], size=docs[0])
        if docs[2] is not None:
            lens[docs[2]] = 0                     # an empty document
        lens[-1] += T - lens.sum()
        assert lens.min() >= 0
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    else:
        cu = np.array([0, T], np.int32)
    rng = np.random.default_rng(17 + kp)
    sel, cu_pools = _synth_pools(rng, cu, kp, Kp)
    mi = W.make_mla_inputs(T, seed=9)
    q, kv = mi.q.to(dev), mi.kv.to(dev)
    sel_d = torch.from_numpy(sel).to(dev)
    cu_d = torch.from_numpy(cu).to(dev) if docs else None
    cp_d = torch.from_numpy(cu_pools).to(dev) if docs else None
    o1, l1 = K.kpool_sparse_mla_fwd_pools(q, kv, sel_d, kp, index_topk, mi.scale, cu_d, cp_d,
                                          always_select_tail=tail)
    tok = K.kpool_expand_indices(sel_d, kp, index_topk, tail, cu_d, cp_d)
    o2, l2 = K.kpool_sparse_mla_fwd(q, kv, tok, mi.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    rows = W.sample_rows(T, n_sample=48, edge=6, seed=kp).numpy()
    tok_ref = ora.expand_rows(sel[rows], cu if docs else None, T, kp, Kp, tail, rows)
    assert np.array_equal(tok_ref, tok.cpu().numpy()[rows])
    check_attn(ora, mi.q, mi.kv, tok_ref, rows, mi.scale, o1.cpu()[rows], l1.cpu()[rows], "pools")


def test_fused_expansion_positioned(K, ora):
    """Decode and chunk rows (kpool_sparse_mla_fwd_pools_at) against the
    explicit tokens of kpool_expand_indices_at, bit for bit, and the oracle."""
    dev = torch.device("cuda")
    kp, index_topk = 4, 256
    Kp = index_topk // kp
    lens_k = np.array([1500, 3100, 77, 2048], np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    nq = np.array([1, 40, 1, 8], np.int32)                # decode and chunk rows
    cu_q = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q_pos = (lens_k - nq).astype(np.int32)
    cu_pools = np.concatenate([[0], np.cumsum(lens_k // kp)]).astype(np.int32)
    rng = np.random.default_rng(23)
    Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
    sel = np.full((Tq, Kp), -1, np.int32)
    for d in range(len(nq)):
        for i in range(nq[d]):
            tau = q_pos[d] + i
            nc = min((tau + 1) // kp, cu_pools[d + 1] - cu_pools[d])
            n = min(nc, Kp)
            sel[cu_q[d] + i, :n] = np.sort(rng.choice(nc, size=n, replace=False)) + cu_pools[d]
    mi = W.make_mla_inputs(Tq, Tk, seed=13)
    args = [torch.from_numpy(a).to(dev) for a in (cu_q, q_pos, cu_k, cu_pools)]
    sel_d = torch.from_numpy(sel).to(dev)
    q, kv = mi.q.to(dev), mi.kv.to(dev)
    o1, l1 = K.kpool_sparse_mla_fwd_pools_at(q, kv, sel_d, kp, index_topk, mi.scale, *args)
    tok = K.kpool_expand_indices_at(sel_d, kp, index_topk, *args)
    o2, l2 = K.kpool_sparse_mla_fwd(q, kv, tok, mi.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    rows = np.arange(Tq)
    tok_ref = ora.expand_rows_at(sel, cu_q, q_pos, cu_k, kp, Kp, True, rows)
    assert np.array_equal(tok_ref, tok.cpu().numpy())
    check_attn(ora, mi.q, mi.kv, tok_ref, rows, mi.scale, o1.cpu(), l1.cpu(), "at")


def test_degenerate_calls(K):
    """T = 0 enqueues nothing; W = 0 and all -1 rows give o = 0, lse = -inf;
    out-of-range indices are skipped; one key token gives o = that row."""
    dev = torch.device("cuda")
    mi = W.make_mla_inputs(3, 5, seed=2)
    q, kv = mi.q.to(dev), mi.kv.to(dev)
    o, lse = K.kpool_sparse_mla_fwd(q[:0], kv, torch.zeros(0, 4, dtype=torch.int32, device=dev), 0.1)
    assert o.shape == (0, H, DC)
    o, lse = K.kpool_sparse_mla_fwd(q, kv, torch.zeros(3, 0, dtype=torch.int32, device=dev), 0.1)
    torch.cuda.synchronize()
    assert torch.all(o.float() == 0) and torch.all(torch.isneginf(lse))
    tok = torch.tensor([[-1, -1, 99, -5], [2, -1, 7, -1], [4, 4, 4, 4]], dtype=torch.int32, device=dev)
    o, lse = K.kpool_sparse_mla_fwd(q, kv, tok, 0.1)
    torch.cuda.synchronize()
    assert torch.all(o[0].float() == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.equal(o[1].view(torch.int16), kv[2].expand(H, DC).view(torch.int16))
    assert torch.equal(o[2].view(torch.int16), kv[4].expand(H, DC).view(torch.int16))
    s = (q[2].float() @ kv[4].float()) * 0.1
    assert torch.allclose(lse[2] - math.log(4.0), s, rtol=1e-5, atol=1e-5)


def test_rejected_shapes(K):
    dev = torch.device("cuda")
    q = torch.zeros(2, 32, 512, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(4, 512, dtype=torch.bfloat16, device=dev)
    tok = torch.zeros(2, 3, dtype=torch.int32, device=dev)
    with pytest.raises(K.KPoolError):
        K.kpool_sparse_mla_fwd(q, kv, tok, 0.1)
    q = torch.zeros(2, 64, 512, dtype=torch.bfloat16, device=dev)
    with pytest.raises(K.KPoolError):
        K.kpool_sparse_mla_fwd(q, kv, tok, 0.0)


@pytest.mark.parametrize("name", ["mla_32k", "mla_thd_32k"])
def test_fullsize_sampled(K, ora, name):
    """The bench's sparse-attention workloads at full size, on the indexer's
    own selection: sampled rows against the oracle; clean status word."""
    dev = torch.device("cuda")
    wl = W.MLA_WORKLOADS[name]
    inp = W.make_inputs(wl, seed=wl.seed)
    cu_d = cp_d = P = None
    cu_h = None
    if wl.n_docs > 1:
        cp_h, P = K.kpool_num_pools(inp.cu_seqlens, wl.T, wl.kpool)
        cu_d, cp_d = inp.cu_seqlens.to(dev), cp_h.to(dev)
        cu_h = inp.cu_seqlens.numpy()
    _, pool_idx, _ = K.kpool_indexer_forward(inp.q.to(dev), inp.k.to(dev), inp.gate.to(dev),
                                             inp.ape.to(dev), inp.w.to(dev), wl.kpool,
                                             wl.index_topk, wl.tail, cu_d, cp_d, P)
    mi = W.make_mla_inputs(wl.T, seed=wl.seed)
    ws = torch.zeros(K.kpool_sparse_mla_workspace_size(), dtype=torch.uint8, device=dev)
    o, lse = K.kpool_sparse_mla_fwd_pools(mi.q.to(dev), mi.kv.to(dev), pool_idx, wl.kpool,
                                          wl.index_topk, mi.scale, cu_d, cp_d, wl.tail, workspace=ws)
    torch.cuda.synchronize()
    assert K.kpool_read_status(ws) == 0
    rows = W.sample_rows(wl.T, n_sample=16, edge=4, seed=3).numpy()
    sel = pool_idx.cpu().numpy()[rows]
    tok = ora.expand_rows(sel, cu_h, wl.T, wl.kpool, wl.Kp, wl.tail, rows)
    check_attn(ora, mi.q, mi.kv, tok, rows, mi.scale, o.cpu()[rows], lse.cpu()[rows], name)


@pytest.mark.parametrize("limit_ns", [1, 3000])
def test_expired_waits(K, ora, limit_ns):
    """With the wait limit lowered the call reports KPOOL_STATUS_TIMEOUT (1 ns)
    or finishes; either way the next call at the default limit is clean and
    matches the oracle."""
    dev = torch.device("cuda")
    T, Tk, Wd = 600, 4000, 1000
    mi = W.make_mla_inputs(T, Tk, seed=21)
    rng = np.random.default_rng(5)
    tok = _random_lists(rng, T, Tk, Wd, [1000, 800, 0, 129], holes=False)
    q, kv, tok_d = mi.q.to(dev), mi.kv.to(dev), torch.from_numpy(tok).to(dev)
    ws = torch.zeros(K.kpool_sparse_mla_workspace_size(), dtype=torch.uint8, device=dev)
    prev = K.kpool_debug_set_wait_limit_ns(limit_ns)
    try:
        assert prev == 2_000_000_000
        K.kpool_sparse_mla_fwd(q, kv, tok_d, mi.scale, workspace=ws)
        torch.cuda.synchronize()
        st = K.kpool_read_status(ws)
    finally:
        assert K.kpool_debug_set_wait_limit_ns(0) == limit_ns
    if limit_ns == 1:
        assert st & K.STATUS_TIMEOUT, st
    o, lse = K.kpool_sparse_mla_fwd(q, kv, tok_d, mi.scale, workspace=ws)
    torch.cuda.synchronize()
    assert K.kpool_read_status(ws) == 0
    rows = np.array([0, 1, 2, 3, 301, 599])
    check_attn(ora, mi.q, mi.kv, tok[rows], rows, mi.scale, o.cpu()[rows], lse.cpu()[rows], "wl")
