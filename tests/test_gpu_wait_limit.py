"""The expired-wait path of the scoring kernel, exercised on purpose.

Every wait inside kpool_score_topk's pipeline (tile info, q tile, pooled-key
stages, accumulators) is bounded; when one runs out the kernel sets
KPOOL_STATUS_TIMEOUT in the call's status word, its CTA's roles stop
waiting, let their in-flight copies and MMAs land, free their tensor memory
and exit.  kpool_debug_set_wait_limit_ns lowers the limit for the launches
that follow so that waits expire at once (1 ns) or part way through (a few
microseconds); afterwards the default is restored and a normal call must
report a clean status and results equal to the oracle's.  No kernel is made
to fault or hang: every wait still ends, and the CTA's epilogue warps leave
their loop together at a barrier they all reach."""
import numpy as np
import pytest
import torch

from sparse_attention_kpool_compress_gb300 import workloads as W
from kpool_checks import check_selection

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_kpool_compress_gb300 as K
    return K


def _clean_call_matches_oracle(K, ora, q, w, pk, pkb, inp, wl, ws, rows):
    idx, sc = K.kpool_score_topk(q, w, pk, wl.kpool, wl.index_topk, workspace=ws)
    torch.cuda.synchronize()
    assert K.kpool_read_status(ws) == 0
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    check_selection(ora, ops, None, wl.kpool, wl.Kp, rows, idx.cpu().numpy()[rows],
                    sc.cpu().numpy()[rows], 1e-3, wl.name)


@pytest.mark.parametrize("limit_ns", [1, 3000])
def test_expired_waits_set_timeout_and_next_call_is_clean(K, ora, limit_ns):
    wl = W.Workload("wl", T=8192, H=64, D=128, kpool=4, index_topk=512)
    inp = W.make_inputs(wl, seed=51)
    dev = torch.device("cuda")
    q, w = inp.q.to(dev), inp.w.to(dev)
    pkb = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(), None, wl.kpool)
    pk = torch.from_numpy(pkb.view(np.int16)).view(torch.bfloat16).to(dev)
    ws = K.new_workspace(wl.T, wl.H, 1, dev)
    prev = K.kpool_debug_set_wait_limit_ns(limit_ns)
    try:
        assert prev == 2_000_000_000
        for _ in range(3):
            K.kpool_score_topk(q, w, pk, wl.kpool, wl.index_topk, workspace=ws)
            torch.cuda.synchronize()
            if K.kpool_read_status(ws) & K.STATUS_TIMEOUT:
                break
        st = K.kpool_read_status(ws)
    finally:
        assert K.kpool_debug_set_wait_limit_ns(0) == limit_ns
    if limit_ns == 1:
        assert st & K.STATUS_TIMEOUT, st
    assert not st & K.STATUS_BAD_SEQLENS
    # the context is intact: the default limit gives a clean, correct result
    rows = W.sample_rows(wl.T, n_sample=256, edge=16).numpy()
    _clean_call_matches_oracle(K, ora, q, w, pk, pkb, inp, wl, ws, rows)


def test_expired_waits_in_the_split_schedule(K, ora):
    """Decode-like call on the split-pool schedule (units on different CTAs,
    the last one merging): with 1 ns waits the call reports a timeout; with
    the default it matches the unsplit schedule bit for bit."""
    wl = W.Workload("wls", T=32768, H=64, D=128, kpool=4, index_topk=512)
    inp = W.make_inputs(wl, seed=52)
    dev = torch.device("cuda")
    pkb = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(), None, wl.kpool)
    pk = torch.from_numpy(pkb.view(np.int16)).view(torch.bfloat16).to(dev)
    n = 8                                           # 8 queries at the end of the sequence
    q, w = inp.q[-n:].to(dev), inp.w[-n:].to(dev)
    cq = torch.tensor([0, n], dtype=torch.int32, device=dev)
    qp = torch.tensor([wl.T - n], dtype=torch.int32, device=dev)
    cp = torch.tensor([0, wl.T // wl.kpool], dtype=torch.int32, device=dev)
    ws = K.new_workspace(n, wl.H, 1, dev, wl.kpool, wl.index_topk)
    prev = K.kpool_debug_set_wait_limit_ns(1)
    try:
        K.kpool_score_topk_at(q, w, pk, wl.kpool, wl.index_topk, cq, qp, cp, workspace=ws)
        torch.cuda.synchronize()
        st = K.kpool_read_status(ws)
    finally:
        K.kpool_debug_set_wait_limit_ns(prev)
    assert st & K.STATUS_TIMEOUT, st
    a_idx, a_sc = K.kpool_score_topk_at(q, w, pk, wl.kpool, wl.index_topk, cq, qp, cp,
                                        workspace=ws)
    torch.cuda.synchronize()
    assert K.kpool_read_status(ws) == 0
    ws1 = K.new_workspace(n, wl.H, 1, dev)          # too small to split: unsplit schedule
    b_idx, b_sc = K.kpool_score_topk_at(q, w, pk, wl.kpool, wl.index_topk, cq, qp, cp,
                                        workspace=ws1)
    torch.cuda.synchronize()
    assert K.kpool_read_status(ws1) == 0
    assert torch.equal(a_idx, b_idx) and torch.equal(a_sc, b_sc)
