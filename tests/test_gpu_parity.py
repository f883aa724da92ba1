"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs.  Bars: pooled keys within 1 BF16 ulp; scores within
1e-3 * S (S = sum_h |w| relu(q.pk)); selections identical except near-tie
swaps; expansion bit-exact.  See tests/kpool_checks.py."""
import math

import numpy as np
import pytest
import torch

from sparse_attention_kpool_compress_gb300 import workloads as W
from kpool_checks import (bf16_bits, bf16_ulp_distance, check_dense_scores, check_pooled_keys,
                          check_selection)

pytestmark = pytest.mark.gpu

TOL = 1e-3
TOL_FP8 = 5e-2


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_kpool_compress_gb300 as K
    K.kpool_version()
    return K


def dev(x):
    return x.to("cuda", non_blocking=False).contiguous()


def bf16_from_bits(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def docs_dev(inp, K):
    cu = inp.cu_seqlens
    if cu.numel() == 2:
        return None, None, inp.wl.T // inp.wl.kpool
    cu_pools, total = K.kpool_num_pools(cu, inp.wl.T, inp.wl.kpool)
    return dev(cu), dev(cu_pools), total


def ora_cu(inp):
    return inp.cu_seqlens.numpy() if inp.cu_seqlens.numel() > 2 else None


def run_compress(K, inp, fp8=False):
    cu, cp, P = docs_dev(inp, K)
    return K.kpool_compress(dev(inp.k), dev(inp.gate), dev(inp.ape), inp.wl.kpool, cu, cp, P,
                            fp8=fp8)


# ---------------------------------------------------------------------------
# compression
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "single_8k", "thd_32k"])
def test_compress_within_one_ulp(K, ora, name):
    inp = W.make_inputs(W.WORKLOADS[name])
    pk = run_compress(K, inp)
    torch.cuda.synchronize()
    want, exact, cond = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(),
                                     ora_cu(inp), inp.wl.kpool, want_cond=True)
    got = bf16_bits(pk)
    check_pooled_keys(got, want, exact, cond, name)
    assert (bf16_ulp_distance(got, want) > 0).mean() < 1e-3


@pytest.mark.parametrize("kp,D,T", [(1, 32, 64), (2, 64, 200), (3, 128, 301), (8, 128, 512),
                                    (16, 64, 1000)])
def test_compress_shapes(K, ora, kp, D, T):
    wl = W.Workload("c", T=T, H=4, D=D, kpool=kp, index_topk=kp * 4)
    inp = W.make_inputs(wl, seed=kp)
    pk = run_compress(K, inp)
    torch.cuda.synchronize()
    want, exact, cond = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(), None, kp,
                                     want_cond=True)
    check_pooled_keys(bf16_bits(pk), want, exact, cond)


def test_compress_thd_with_empty_and_short_docs(K, ora):
    T, D, kp = 400, 64, 4
    wl = W.Workload("c", T=T, H=4, D=D, kpool=kp, index_topk=16)
    inp = W.make_inputs(wl, seed=3)
    cu = torch.tensor([0, 0, 3, 10, 10, 211, 400], dtype=torch.int32)
    cu_pools, P = K.kpool_num_pools(cu, T, kp)
    pk = K.kpool_compress(dev(inp.k), dev(inp.gate), dev(inp.ape), kp, dev(cu), dev(cu_pools), P)
    torch.cuda.synchronize()
    want, exact, cond = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(),
                                     cu.numpy(), kp, want_cond=True)
    assert P == want.shape[0]
    check_pooled_keys(bf16_bits(pk), want, exact, cond)


# ---------------------------------------------------------------------------
# FP8 input emulation
# ---------------------------------------------------------------------------

def _fp8_compare(ora, x_bits, codes, scales):
    oc, osc, y, b = ora.fp8_rows(x_bits, want_intermediate=True)
    codes = codes.reshape(oc.shape)
    scales = scales.reshape(osc.shape)
    row_bad = np.where((codes != oc).any(axis=1) | (scales != osc))[0]
    # A mismatch is only allowed where the FP32 rotation lands next to a BF16
    # rounding midpoint (the oracle rotates exactly): check that every
    # differing row has an element within 2^-20 relative of a midpoint.
    for r in row_bad:
        yb = y[r]
        bits = np.array([ora.bf16_from_double(v) for v in yb], np.uint16)
        lo = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ulp = np.abs(lo) * 2.0 ** -7 + 1e-300
        frac = np.abs(np.abs(yb - lo) / ulp - 0.5)
        assert (frac < 2.0 ** -12).any(), "row %d differs without a near-midpoint element" % r
    return len(row_bad)


def test_quantize_fp8_matches_oracle(K, ora):
    gen = torch.Generator().manual_seed(11)
    x = torch.randn(4096, 128, generator=gen).to(torch.bfloat16)
    x[5] = 0
    x[6] *= 1e-30
    x[7] *= 1e30
    codes, sc = K.kpool_quantize_fp8(dev(x))
    torch.cuda.synchronize()
    nbad = _fp8_compare(ora, W.bits(x), codes.cpu().numpy(), sc.cpu().numpy())
    assert nbad <= 8
    assert float(sc[5]) == 1.0 and int(codes[5].abs().sum()) == 0


def test_quantize_fp8_ragged_rows(K):
    """Row counts that do not fill the last warp: the same codes as the full
    call, and nothing written past the last row."""
    gen = torch.Generator().manual_seed(13)
    x = dev(torch.randn(4096, 128, generator=gen).to(torch.bfloat16))
    full_c, full_s = K.kpool_quantize_fp8(x)
    B = K.binding
    for rows in (4093, 4089, 1):
        c = torch.full((4096, 128), 0xAB, dtype=torch.uint8, device=x.device)
        sc = torch.full((4096,), 7.0, dtype=torch.float32, device=x.device)
        rc = B._lib.kpool_quantize_fp8(B._ptr(x), rows, 128, B._ptr(c), B._ptr(sc),
                                       B._stream(x.device))
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.equal(c[:rows], full_c[:rows]) and torch.equal(sc[:rows], full_s[:rows])
        assert bool((c[rows:] == 0xAB).all()) and bool((sc[rows:] == 7.0).all())


def test_compress_fp8_matches_oracle(K, ora):
    wl = W.Workload("f", T=4096, H=4, D=128, kpool=4, index_topk=64)
    inp = W.make_inputs(wl, seed=12)
    pk, pk8, pks = run_compress(K, inp, fp8=True)
    torch.cuda.synchronize()
    want, exact, cond = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(), None, 4,
                                     want_cond=True)
    got = bf16_bits(pk)
    check_pooled_keys(got, want, exact, cond)
    same = (got == want).all(axis=1)
    # compare FP8 of the rows whose bf16 pooled key agrees exactly
    nbad = _fp8_compare(ora, got[same], pk8.cpu().numpy()[same], pks.cpu().numpy()[same])
    assert nbad <= 4


# ---------------------------------------------------------------------------
# scoring (oracle pooled keys fed to both sides: accumulation order only)
# ---------------------------------------------------------------------------

def _ora_pk(ora, inp):
    return ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(), ora_cu(inp),
                        inp.wl.kpool)


@pytest.mark.parametrize("name,nrows", [("tiny", None), ("single_8k", 384)])
def test_score_dense(K, ora, name, nrows):
    inp = W.make_inputs(W.WORKLOADS[name])
    wl = inp.wl
    pkb = _ora_pk(ora, inp)
    cu, cp, P = docs_dev(inp, K)
    out = K.kpool_score_dense(dev(inp.q), dev(inp.w), dev(bf16_from_bits(pkb)), wl.kpool, cu, cp)
    torch.cuda.synchronize()
    rows = np.arange(wl.T) if nrows is None else W.sample_rows(wl.T, nrows, 32).numpy()
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    osc, ocd = ora.score_rows_full(ops, ora_cu(inp), wl.kpool, rows)
    check_dense_scores(out.cpu().numpy()[rows], osc, ocd, TOL, name)


@pytest.mark.parametrize("name", ["tiny", "single_8k", "thd_32k"])
def test_score_topk_selection(K, ora, name):
    inp = W.make_inputs(W.WORKLOADS[name])
    wl = inp.wl
    pkb = _ora_pk(ora, inp)
    cu, cp, P = docs_dev(inp, K)
    idx, sc = K.kpool_score_topk(dev(inp.q), dev(inp.w), dev(bf16_from_bits(pkb)), wl.kpool,
                                 wl.index_topk, cu, cp)
    torch.cuda.synchronize()
    rows = np.arange(wl.T)
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    st = check_selection(ora, ops, ora_cu(inp), wl.kpool, wl.Kp, rows, idx.cpu().numpy(),
                         sc.cpu().numpy(), TOL, name)
    assert st["swaps"] <= max(2, wl.T // 1000)


@pytest.mark.parametrize("H", [4, 8, 16, 32, 64, 128])
def test_score_topk_heads(K, ora, H):
    wl = W.Workload("h", T=700, H=H, D=64, kpool=4, index_topk=40)
    inp = W.make_inputs(wl, seed=H)
    pkb = _ora_pk(ora, inp)
    idx, sc = K.kpool_score_topk(dev(inp.q), dev(inp.w), dev(bf16_from_bits(pkb)), 4, 40)
    torch.cuda.synchronize()
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    check_selection(ora, ops, None, 4, 10, np.arange(wl.T), idx.cpu().numpy(), sc.cpu().numpy(),
                    TOL, "H%d" % H)


@pytest.mark.parametrize("kp,D,T,topk", [(1, 32, 300, 16), (2, 128, 1030, 64), (3, 64, 777, 30),
                                         (8, 128, 2100, 256), (4, 32, 5, 8), (4, 128, 3, 8)])
def test_score_topk_shapes(K, ora, kp, D, T, topk):
    wl = W.Workload("s", T=T, H=16, D=D, kpool=kp, index_topk=topk)
    inp = W.make_inputs(wl, seed=kp + D)
    pkb = _ora_pk(ora, inp)
    pk = dev(bf16_from_bits(pkb)) if pkb.shape[0] else torch.empty(0, D, dtype=torch.bfloat16,
                                                                    device="cuda")
    idx, sc = K.kpool_score_topk(dev(inp.q), dev(inp.w), pk, kp, topk)
    torch.cuda.synchronize()
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    check_selection(ora, ops, None, kp, topk // kp, np.arange(T), idx.cpu().numpy(),
                    sc.cpu().numpy(), TOL, "shape")


def test_score_topk_thd_empty_docs(K, ora):
    T, H, D, kp, topk = 2000, 32, 128, 4, 64
    wl = W.Workload("e", T=T, H=H, D=D, kpool=kp, index_topk=topk)
    inp = W.make_inputs(wl, seed=21)
    cu = torch.tensor([0, 0, 2, 9, 9, 600, 601, 1500, 2000], dtype=torch.int32)
    pkb = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(), cu.numpy(), kp)
    cu_pools, P = K.kpool_num_pools(cu, T, kp)
    idx, sc = K.kpool_score_topk(dev(inp.q), dev(inp.w), dev(bf16_from_bits(pkb)), kp, topk,
                                 dev(cu), dev(cu_pools))
    torch.cuda.synchronize()
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    check_selection(ora, ops, cu.numpy(), kp, topk // kp, np.arange(T), idx.cpu().numpy(),
                    sc.cpu().numpy(), TOL, "thd-empty")


def test_ties_lowest_index(K):
    """All-zero q: every score is 0, so every row keeps its lowest pools."""
    T, H, D, kp, topk = 3000, 64, 128, 4, 256
    q = torch.zeros(T, H, D, dtype=torch.bfloat16, device="cuda")
    w = torch.randn(T, H, device="cuda")
    pk = torch.randn(T // kp, D, device="cuda").to(torch.bfloat16)
    idx, sc = K.kpool_score_topk(q, w, pk, kp, topk)
    torch.cuda.synchronize()
    idx = idx.cpu().numpy()
    Kp = topk // kp
    for t in range(T):
        n = min((t + 1) // kp, Kp)
        assert np.array_equal(idx[t, :n], np.arange(n)), t
        assert np.all(idx[t, n:] == -1)
    assert torch.all(sc[sc > -math.inf] == 0)


def test_identical_keys_tie(K, ora):
    T, H, D, kp, topk = 2048, 64, 128, 4, 128
    wl = W.Workload("i", T=T, H=H, D=D, kpool=kp, index_topk=topk)
    inp = W.make_inputs(wl, seed=5)
    pkb = _ora_pk(ora, inp)
    pkb[100:300] = pkb[100]      # many equal pooled keys
    idx, sc = K.kpool_score_topk(dev(inp.q), dev(inp.w), dev(bf16_from_bits(pkb)), kp, topk)
    torch.cuda.synchronize()
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    check_selection(ora, ops, None, kp, topk // kp, np.arange(0, T, 7), idx.cpu().numpy()[::7],
                    sc.cpu().numpy()[::7], TOL, "ident")


def test_fp8_scoring_matches_oracle_on_same_codes(K, ora):
    T, H, kp, topk = 3000, 64, 4, 256
    wl = W.Workload("f", T=T, H=H, D=128, kpool=kp, index_topk=topk)
    inp = W.make_inputs(wl, seed=8)
    pkb = _ora_pk(ora, inp)
    qc, qs = ora.fp8_rows(W.bits(inp.q).reshape(-1, 128))
    pc, ps = ora.fp8_rows(pkb)
    qc = qc.reshape(T, H, 128)
    qs = qs.reshape(T, H)
    idx, sc = K.kpool_score_topk(dev(torch.from_numpy(qc)), dev(inp.w), dev(torch.from_numpy(pc)),
                                 kp, topk, q_scale=dev(torch.from_numpy(qs)),
                                 pk_scale=dev(torch.from_numpy(ps)))
    torch.cuda.synchronize()
    ops = ora.Operands(qc, inp.w.numpy(), pc, qs, ps)
    check_selection(ora, ops, None, kp, topk // kp, np.arange(T), idx.cpu().numpy(),
                    sc.cpu().numpy(), TOL, "fp8-same-codes")


# ---------------------------------------------------------------------------
# expansion
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "single_8k", "thd_32k"])
@pytest.mark.parametrize("tail", [True, False])
def test_expand_bit_exact(K, ora, name, tail):
    inp = W.make_inputs(W.WORKLOADS[name])
    wl = inp.wl
    pkb = _ora_pk(ora, inp)
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    rows = np.arange(wl.T) if wl.T <= 8192 else W.sample_rows(wl.T, 1024).numpy()
    o = ora.select_rows(ops, ora_cu(inp), wl.kpool, wl.Kp, rows)
    sel = np.full((wl.T, wl.Kp), -1, np.int32)
    sel[rows] = o["sel"]
    cu, cp, P = docs_dev(inp, K)
    tok = K.kpool_expand_indices(dev(torch.from_numpy(sel)), wl.kpool, wl.index_topk, tail, cu, cp)
    torch.cuda.synchronize()
    want = ora.expand_rows(o["sel"], ora_cu(inp), wl.T, wl.kpool, wl.Kp, tail, rows)
    assert np.array_equal(tok.cpu().numpy()[rows], want)


@pytest.mark.parametrize("kp", [1, 2, 3, 4, 5, 8, 16])
def test_expand_kpool_values(K, ora, kp):
    T, Kp = 500, 7
    cu = np.array([0, 3, 130, 131, 500], np.int32)
    cp = ora.cu_pools(cu, kp)
    rng = np.random.default_rng(kp)
    sel = np.full((T, Kp), -1, np.int32)
    for t in range(T):
        d = np.searchsorted(cu, t, side="right") - 1
        nc = (t - cu[d] + 1) // kp
        n = min(nc, Kp)
        sel[t, :n] = np.sort(rng.choice(nc, n, replace=False)) + cp[d] if n else []
    tok = K.kpool_expand_indices(dev(torch.from_numpy(sel)), kp, Kp * kp, True,
                                 dev(torch.from_numpy(cu)), dev(torch.from_numpy(cp)))
    torch.cuda.synchronize()
    want = ora.expand_rows(sel, cu, T, kp, Kp, True, np.arange(T))
    assert np.array_equal(tok.cpu().numpy(), want)


# ---------------------------------------------------------------------------
# whole path (GPU compress -> score/top-k -> expand)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "single_8k"])
def test_pipeline_end_to_end(K, ora, name):
    inp = W.make_inputs(W.WORKLOADS[name])
    wl = inp.wl
    cu, cp, P = docs_dev(inp, K)
    tok, idx, sc = K.kpool_indexer_forward(dev(inp.q), dev(inp.k), dev(inp.gate), dev(inp.ape),
                                           dev(inp.w), wl.kpool, wl.index_topk, True, cu, cp, P)
    torch.cuda.synchronize()
    pkb = _ora_pk(ora, inp)
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    rows = np.arange(wl.T)
    idx_h = idx.cpu().numpy()
    check_selection(ora, ops, ora_cu(inp), wl.kpool, wl.Kp, rows, idx_h, sc.cpu().numpy(),
                    TOL, name)
    want = ora.expand_rows(idx_h, ora_cu(inp), wl.T, wl.kpool, wl.Kp, True, rows)
    assert np.array_equal(tok.cpu().numpy(), want)


def test_status_clean_and_bad_seqlens(K):
    T, H, D = 256, 64, 128
    q = torch.randn(T, H, D, device="cuda").to(torch.bfloat16)
    w = torch.randn(T, H, device="cuda")
    pk = torch.randn(T // 4, D, device="cuda").to(torch.bfloat16)
    ws = K.new_workspace(T, H, 2)
    K.kpool_score_topk(q, w, pk, 4, 32, workspace=ws)
    assert K.kpool_read_status(ws) == 0
    cu = torch.tensor([0, 200, 100], dtype=torch.int32, device="cuda")   # decreasing, last != T
    cp = torch.tensor([0, 50, 25], dtype=torch.int32, device="cuda")
    K.kpool_score_topk(q, w, pk, 4, 32, cu, cp, workspace=ws)
    assert K.kpool_read_status(ws) & K.STATUS_BAD_SEQLENS


def test_fp8_chain_hand_worked_onehot_gpu(K):
    """kpool_quantize_fp8 on the one-hot rows of tests/golden/fp8_onehot_worked.txt:
    the hand-worked codes and scales, including an exact E4M3 tie; and the same
    rows as pooled keys (a pool of identical keys compresses to that key)."""
    from test_oracle_pins import _fp8_onehot_cases, _fp8_onehot_expected
    cases = _fp8_onehot_cases()
    x = torch.zeros(len(cases), 128, dtype=torch.float32)
    for r, (v, j, _, _, _) in enumerate(cases):
        x[r, j] = v
    xb = x.to(torch.bfloat16)
    codes, scales = K.kpool_quantize_fp8(dev(xb))
    # pooled keys: kpool = 2, both slots of pool r hold row r
    k = xb.repeat_interleave(2, dim=0)
    _, pk8, pks = K.kpool_compress(dev(k), dev(torch.zeros_like(k)), dev(torch.zeros(2, 128)), 2,
                                   fp8=True)
    torch.cuda.synchronize()
    for got_c, got_s in ((codes.cpu().numpy(), scales.cpu().numpy()),
                         (pk8.cpu().numpy(), pks.cpu().numpy())):
        for r, (v, j, e, cpos, cneg) in enumerate(cases):
            assert got_s[r] == 2.0 ** e, (v, j, got_s[r])
            assert np.array_equal(got_c[r], _fp8_onehot_expected(v, j, cpos, cneg)), (v, j)


def test_score_and_selection_hand_worked_gpu(K):
    """tests/golden/score_select_worked.txt padded to H = 4 (w = 0 on the extra
    heads) and D = 32 (zeros): the hand-worked scores, selections and the tie to
    the lower pool index, exactly; kpool = 1 so pk = k and tokens = pools."""
    from test_oracle_pins import score_select_worked
    q, k, w, want_idx, want_sc = score_select_worked(pad_heads=4, pad_dims=32)
    pk = K.kpool_compress(dev(k), dev(torch.zeros_like(k)), dev(torch.zeros(1, 32)), 1)
    idx, sc = K.kpool_score_topk(dev(q), dev(w), pk, 1, 2)
    tok = K.kpool_expand_indices(idx, 1, 2, True)
    torch.cuda.synchronize()
    assert torch.equal(pk.cpu(), k)
    assert np.array_equal(idx.cpu().numpy(), want_idx)
    assert np.array_equal(sc.cpu().numpy().astype(np.float64), want_sc)
    assert np.array_equal(tok.cpu().numpy(), want_idx)


@pytest.mark.parametrize("kp", [2, 3, 4])
@pytest.mark.parametrize("D", [32, 128])
def test_compress_hand_worked_moderate_logits_gpu(K, kp, D):
    """kpool_compress on the hand-worked pools of tests/golden/compress_worked.txt
    (softmax weights 1/4, 3/4, 1/8, 0.1 .. 0.4 at moderate logits): the pooled
    keys equal the hand-derived BF16 values exactly, on the plain and on the
    FP8-output path (whose BF16 pooled key is the same)."""
    from test_oracle_pins import compress_worked_inputs
    kb, gb, ape, want = compress_worked_inputs(kp, D)
    pk = K.kpool_compress(dev(kb), dev(gb), dev(torch.from_numpy(ape)), kp)
    torch.cuda.synchronize()
    assert np.array_equal(pk.float().cpu().numpy()[0].astype(np.float64), want)
    if D == 128:
        pk2, _, _ = K.kpool_compress(dev(kb), dev(gb), dev(torch.from_numpy(ape)), kp, fp8=True)
        torch.cuda.synchronize()
        assert torch.equal(pk2.cpu(), pk.cpu())
