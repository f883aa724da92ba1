"""Pins for the CPU oracle: each function is checked against something other
than itself -- number-format definitions enumerated exhaustively, library
routines (torch's bf16/E4M3 casts, scipy's Hadamard matrix, numpy), closed
forms of special cases, invariants, and brute force on tiny inputs.

Sources: Megatron-LM PR "GLM5.3 Flash (KDA + mHC + KPool DSA) support + FP8"
(Changes section 3; Testing: test_kpool_causal_tail), SkyRL PR
"GLM-5.3-Flash (glm5_next) Megatron support" (commit "k-pool indexer"),
xtuner PR "GLM-5.3-Flash F5: NoPE DSA + KPool indexer" (relu homogeneity).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

from sparse_attention_kpool_compress_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits_of(x_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_val(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def test_bf16_rounding_matches_torch(ora):
    """Oracle double->bf16 RNE equals torch's float32->bf16 cast (a library
    routine) on float32 inputs, incl. exact ties, subnormals and overflow."""
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-39).astype(np.float32),     # subnormal range
        np.clip(rng.standard_normal(500) * 3e38, -3.3e38, 3.3e38).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, -3.3895314e38], dtype=np.float32),
    ])
    # exact ties: bf16 value + half an ulp (low 16 bits 0x8000), both parities
    tie_bits = (rng.integers(0x0080, 0x7F00, 2000, dtype=np.uint32) << 16) | 0x8000
    xs = np.concatenate([xs, tie_bits.astype(np.uint32).view(np.float32)])
    want = bf16_bits_of(xs)
    got = np.array([ora.bf16_from_double(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_decode(ora):
    for b in [0x0000, 0x8000, 0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4049]:
        assert ora.bf16_to_double(b) == float(bf16_val(np.array([b], np.uint16))[0])


def _e4m3_table():
    """All finite E4M3 values from the format definition (sign, 4-bit
    exponent with bias 7, 3-bit fraction, exponent 0 subnormal, S.1111.111
    NaN)."""
    vals = {}
    for c in range(256):
        s, E, M = c >> 7, (c >> 3) & 15, c & 7
        if E == 15 and M == 7:
            continue
        v = (M / 8.0) * 2.0 ** -6 if E == 0 else (1 + M / 8.0) * 2.0 ** (E - 7)
        vals[c] = -v if s else v
    return vals


def test_e4m3_decode_matches_definition_and_torch(ora):
    table = _e4m3_table()
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    tv = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c, v in table.items():
        assert ora.e4m3_to_double(c) == v
        assert tv[c] == v
    assert math.isnan(ora.e4m3_to_double(0x7F)) and math.isnan(ora.e4m3_to_double(0xFF))
    assert max(table.values()) == 448.0


def test_e4m3_rounding_exhaustive_over_bf16(ora):
    """Every one of the 2^16 bf16 inputs: the oracle's E4M3 code is the
    nearest finite E4M3 value (ties to the even code), saturated to +-448."""
    table = _e4m3_table()
    pos = sorted((v, c) for c, v in table.items() if c < 0x80)
    pv = np.array([v for v, _ in pos])
    pc = np.array([c for _, c in pos])
    for b in range(1 << 16):
        x = float(bf16_val(np.array([b], np.uint16))[0])
        if math.isnan(x) or math.isinf(x):
            continue
        got = ora.e4m3_from_double(x)
        ax = abs(x)
        if ax >= 448.0:
            want = 0x7E
        else:
            d = np.abs(pv - ax)
            m = d.min()
            cands = pc[d == m]
            want = int(cands[0]) if len(cands) == 1 else int([c for c in cands if c % 2 == 0][0])
        if math.copysign(1.0, x) < 0:
            want |= 0x80
        assert got == want, (hex(b), x, got, want)


def test_e4m3_matches_torch_in_range(ora):
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(3000) * 50, rng.standard_normal(1000) * 1e-2])
    xs = xs[np.abs(xs) < 440].astype(np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([ora.e4m3_from_double(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_pow2_scale_closed_form(ora):
    assert ora.pow2_scale(0.0) == 1.0
    assert ora.pow2_scale(448.0) == 1.0
    assert ora.pow2_scale(448.0 * 1.0001) == 2.0
    assert ora.pow2_scale(224.0) == 0.5
    assert ora.pow2_scale(224.5) == 1.0
    assert ora.pow2_scale(3.5) == 2.0 ** -7
    rng = np.random.default_rng(3)
    for a in np.abs(rng.standard_normal(500)) * 10.0 ** rng.integers(-6, 6, 500):
        s = ora.pow2_scale(float(a))
        assert math.log2(s) == round(math.log2(s))
        assert a <= 448.0 * s and a > 448.0 * s / 2


# ---------------------------------------------------------------------------
# Hadamard / FP8 emulation (Megatron Testing: Hadamard-matrix reference)
# ---------------------------------------------------------------------------

def test_hadamard_matrix_is_sylvester(ora):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    Hm = ora.hadamard_matrix(128)
    assert np.array_equal(Hm, scipy_linalg.hadamard(128).astype(np.float64))
    assert np.array_equal(Hm @ Hm.T, 128 * np.eye(128))


def _fwht(x):
    """Iterative fast Walsh-Hadamard transform (natural order), float64."""
    y = x.copy()
    h = 1
    n = y.shape[-1]
    while h < n:
        y = y.reshape(*y.shape[:-1], n // (2 * h), 2, h)
        a, b = y[..., 0, :].copy(), y[..., 1, :].copy()
        y[..., 0, :], y[..., 1, :] = a + b, a - b
        y = y.reshape(*y.shape[:-3], n)
        h *= 2
    return y


def test_fp8_rows_matches_fast_wht_chain(ora):
    """y = H x / sqrt(128) equals a fast WHT; b is the bf16 rounding of y; the
    scale is the power of two of max|b|/448; codes are the E4M3 rounding of
    b/s; an all-zero row gets scale 1."""
    gen = torch.Generator().manual_seed(5)
    x = torch.randn(64, 128, generator=gen).to(torch.bfloat16)
    x[3] = 0
    x[7] *= 1000
    xb = W.bits(x)
    codes, scales, y, b = ora.fp8_rows(xb, want_intermediate=True)
    yref = _fwht(bf16_val(xb)) / math.sqrt(128)
    assert np.allclose(y, yref, rtol=1e-14, atol=1e-14)
    # b: nearest bf16 to y (checked through torch on float32(y) where float32(y)
    # is not near a tie; y exact in double to 1e-16 relative)
    bv = bf16_val(b)
    assert np.all(np.abs(bv - y) <= np.abs(y) * 2.0 ** -8 + 1e-45)
    b_t = bf16_bits_of(y.astype(np.float32))
    assert np.mean(b_t == b) > 0.999
    amax = np.abs(bv).max(axis=1)
    for r in range(64):
        assert scales[r] == ora.pow2_scale(float(amax[r]))
    assert scales[3] == 1.0 and np.all(codes[3] == 0)
    deq = np.array([[ora.e4m3_to_double(int(c)) for c in row] for row in codes[:8]])
    for r in range(8):
        want = np.array([ora.e4m3_from_double(v / scales[r]) for v in bv[r]])
        assert np.array_equal(codes[r], want)
        assert np.all(np.abs(deq[r]) <= 448.0)


# ---------------------------------------------------------------------------
# Compression ([MG] section 3, [SK] k-pool commit)
# ---------------------------------------------------------------------------

def _rand_inputs(T, D, kp, seed=0):
    gen = torch.Generator().manual_seed(seed)
    k = torch.randn(T, D, generator=gen).to(torch.bfloat16)
    gate = torch.randn(T, D, generator=gen).to(torch.bfloat16)
    ape = torch.randn(kp, D, generator=gen) * 0.1
    return W.bits(k), W.bits(gate), ape.numpy()


def test_softmax_weights_sum_to_one(ora):
    kb, gb, ape = _rand_inputs(64, 32, 4)
    for first in (0, 4, 60):
        a = ora.pool_weights(gb, ape, first, 4)
        assert np.all(a > 0)
        assert np.allclose(a.sum(axis=0), 1.0, atol=1e-15, rtol=0)


def test_compress_zero_gate_is_mean(ora):
    kb, _, _ = _rand_inputs(64, 32, 4)
    gz = np.zeros_like(kb)
    az = np.zeros((4, 32), np.float32)
    pk = ora.compress(kb, gz, az, None, 4)
    mean = bf16_val(kb).reshape(16, 4, 32).mean(axis=1)
    assert np.array_equal(pk, bf16_bits_of(mean.astype(np.float32)))


def test_compress_identical_keys_and_kp1(ora):
    kb, gb, ape = _rand_inputs(64, 32, 4)
    same = np.repeat(kb[::4], 4, axis=0)
    pk = ora.compress(same, gb, ape, None, 4)
    assert np.array_equal(pk, kb[::4])
    # kpool = 1, any gate: the softmax over one slot is 1 -> pk = k bit-exact
    pk1 = ora.compress(kb, gb, ape[:1], None, 1)
    assert np.array_equal(pk1, kb)


def test_compress_slot_and_dim_indexing(ora):
    """ape[s, d] selects slot s*(d) = d mod kp almost surely (one-hot softmax):
    pk[j, d] must equal k[j*kp + (d mod kp), d].  Catches a transposed ape or
    a wrong slot/token index."""
    T, D, kp = 64, 32, 4
    kb, _, _ = _rand_inputs(T, D, kp, seed=9)
    ape = np.full((kp, D), -40.0, np.float32)
    for d in range(D):
        ape[d % kp, d] = 40.0
    pk = ora.compress(kb, np.zeros_like(kb), ape, None, kp)
    want = np.array([[kb[j * kp + d % kp, d] for d in range(D)] for j in range(T // kp)])
    assert np.array_equal(pk, want)
    # the same selection made through the gate instead of ape
    gf = np.full((T, D), -40.0, np.float32)
    for t in range(T):
        for d in range(D):
            if t % kp == (d + 1) % kp:
                gf[t, d] = 40.0
    pk2 = ora.compress(kb, bf16_bits_of(gf), np.zeros((kp, D), np.float32), None, kp)
    want2 = np.array([[kb[j * kp + (d + 1) % kp, d] for d in range(D)] for j in range(T // kp)])
    assert np.array_equal(pk2, want2)


def test_compress_shift_invariance(ora):
    """Adding a per-dimension constant to every slot's ape leaves the softmax
    (and pk) unchanged.  ape is put on a coarse grid so that the shifted
    float32 values are exact."""
    kb, gb, ape = _rand_inputs(64, 32, 4, seed=4)
    ape = (np.round(ape * 256) / 256).astype(np.float32)
    _, ex1 = ora.compress(kb, gb, ape, None, 4, want_exact=True)
    shift = (np.arange(32) - 16).astype(np.float32) / 8
    ape2 = ape + shift
    assert np.array_equal(ape2.astype(np.float64), ape.astype(np.float64) + shift)
    _, ex2 = ora.compress(kb, gb, ape2, None, 4, want_exact=True)
    assert np.allclose(ex1, ex2, rtol=1e-15, atol=0)


def test_compress_thd_restarts_pools(ora):
    """Packed THD: pools restart at document boundaries; the packed result is
    the per-document results concatenated; partial trailing pools dropped."""
    kb, gb, ape = _rand_inputs(64, 32, 4, seed=6)
    cu = np.array([0, 10, 27, 27, 64], np.int32)   # includes an empty document
    pk = ora.compress(kb, gb, ape, cu, 4)
    parts = [ora.compress(kb[a:b], gb[a:b], ape, None, 4) for a, b in zip(cu[:-1], cu[1:])
             if b - a >= 4] + []
    assert pk.shape[0] == 10 // 4 + 17 // 4 + 0 + 37 // 4
    assert np.array_equal(pk, np.concatenate(parts))
    assert list(ora.cu_pools(cu, 4)) == [0, 2, 6, 6, 15]


# ---------------------------------------------------------------------------
# Scoring and selection
# ---------------------------------------------------------------------------

def _score_inputs(T, H, D, P, seed=0):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(T, H, D, generator=gen).to(torch.bfloat16)
    pk = torch.randn(P, D, generator=gen).to(torch.bfloat16)
    w = torch.randn(T, H, generator=gen) / math.sqrt(H)
    return W.bits(q), W.bits(pk), w.numpy()


def test_kp1_reduces_to_token_level_indexer(ora):
    """kpool=1, gate=0, ape=0: pk = k and the scores are the textbook
    per-token DSA indexer sum_h w * relu(q . k_s) over s <= t (numpy,
    float64).  Tail is always empty."""
    T, H, D = 40, 3, 32
    qb, kb, w = _score_inputs(T, H, D, T, seed=1)
    pk = ora.compress(kb, np.zeros_like(kb), np.zeros((1, D), np.float32), None, 1)
    assert np.array_equal(pk, kb)
    ops = ora.Operands(qb.reshape(T, H, D), w, pk)
    full, _ = ora.score_rows_full(ops, None, 1, np.arange(T))
    qv, kv = bf16_val(qb).reshape(T, H, D), bf16_val(kb)
    ref = np.einsum("th,tsh->ts", w.astype(np.float64),
                    np.maximum(np.einsum("thd,sd->tsh", qv, kv), 0))
    mask = np.tril(np.ones((T, T), bool))
    assert np.allclose(full[mask], ref[mask], rtol=1e-12, atol=1e-12)
    assert np.all(np.isneginf(full[~mask]))
    out = ora.select_rows(ops, None, 1, 8, np.arange(T))
    exp = ora.expand_rows(out["sel"], None, T, 1, 8, True, np.arange(T))
    for t in range(T):
        toks = exp[t][exp[t] >= 0]
        want = np.sort(np.argsort(-ref[t, :t + 1], kind="stable")[:8])
        assert np.array_equal(toks, want)


def test_single_head_unit_weight_is_dot_sort(ora):
    """H=1, w=1: score = relu(q . pk); selection = sort by it (numpy)."""
    T, D, kp, Kp = 64, 32, 2, 5
    qb, pkb, _ = _score_inputs(T, 1, D, T // kp, seed=2)
    w = np.ones((T, 1), np.float32)
    ops = ora.Operands(qb.reshape(T, 1, D), w, pkb)
    full, cond = ora.score_rows_full(ops, None, kp, np.arange(T))
    dots = bf16_val(qb).reshape(T, D) @ bf16_val(pkb).T
    out = ora.select_rows(ops, None, kp, Kp, np.arange(T))
    for t in range(T):
        nc = (t + 1) // kp
        assert np.allclose(full[t, :nc], np.maximum(dots[t, :nc], 0), rtol=1e-13, atol=0)
        assert np.array_equal(cond[t, :nc], full[t, :nc])
        order = sorted(range(nc), key=lambda j: (-max(dots[t, j], 0.0), j))[:Kp]
        sel = out["sel"][t]
        assert np.array_equal(sel[sel >= 0], np.sort(order))


def test_relu_homogeneity(ora):
    """[XT]: scaling q by c > 0 (e.g. head_dim^-0.5) inside the relu equals
    scaling w by c: same selection, scores scaled by c."""
    T, H, D, kp, Kp = 96, 4, 32, 4, 6
    qb, pkb, w = _score_inputs(T, H, D, T // kp, seed=3)
    c = 2.0 ** -3   # exact in bf16 so q*c is representable
    qs = bf16_bits_of((bf16_val(qb) * c).astype(np.float32))
    a = ora.select_rows(ora.Operands(qs.reshape(T, H, D), w, pkb), None, kp, Kp, np.arange(T))
    b = ora.select_rows(ora.Operands(qb.reshape(T, H, D), (w * c).astype(np.float32), pkb),
                        None, kp, Kp, np.arange(T))
    o = ora.select_rows(ora.Operands(qb.reshape(T, H, D), w, pkb), None, kp, Kp, np.arange(T))
    assert np.array_equal(a["sel"], b["sel"]) and np.array_equal(a["sel"], o["sel"])
    fin = np.isfinite(o["sel_score"])
    assert np.allclose(a["sel_score"][fin], c * o["sel_score"][fin], rtol=1e-13, atol=0)


def test_brute_force_subsets(ora):
    """Tiny input: the selected set maximises the score sum over every Kp-subset
    of the causal pools, lexicographically smallest among equal sums; each
    score re-derived by a naive Python loop."""
    T, H, D, kp, Kp = 28, 2, 8, 2, 3
    qb, pkb, w = _score_inputs(T, H, D, T // kp, seed=4)
    ops = ora.Operands(qb.reshape(T, H, D), w, pkb)
    out = ora.select_rows(ops, None, kp, Kp, np.arange(T))
    qv, pv = bf16_val(qb).reshape(T, H, D), bf16_val(pkb)
    for t in range(T):
        nc = (t + 1) // kp
        sc = []
        for j in range(nc):
            s = 0.0
            for h in range(H):
                x = 0.0
                for d in range(D):
                    x += qv[t, h, d] * pv[j, d]
                s += float(w[t, h]) * max(x, 0.0)
            sc.append(s)
        rows, _ = ora.score_pairs(ops, None, kp, [t] * nc, list(range(nc)))
        assert np.allclose(rows, sc, rtol=1e-12, atol=1e-15)
        best = None
        for sub in itertools.combinations(range(nc), min(Kp, nc)):
            key = (-sum(sorted((sc[j] for j in sub), reverse=True)), sub)
            if best is None or key < best:
                best = key
        sel = out["sel"][t]
        assert list(sel[sel >= 0]) == list(best[1]), t


def test_ties_go_to_lower_pool_index(ora):
    """Identical pooled keys tie exactly; a budget that splits them keeps the
    lower pool indices."""
    T, H, D, kp, Kp = 64, 2, 16, 4, 3
    qb, pkb, w = _score_inputs(T, H, D, T // kp, seed=5)
    pkb[:] = pkb[0]
    w = np.abs(w) + 0.1
    out = ora.select_rows(ora.Operands(qb.reshape(T, H, D), w.astype(np.float32), pkb),
                          None, kp, Kp, np.arange(T))
    for t in range(T):
        nc = (t + 1) // kp
        sel = out["sel"][t]
        assert list(sel[sel >= 0]) == list(range(min(nc, Kp)))


def test_condition_scale_bounds_score(ora):
    T, H, D, kp = 48, 4, 16, 4
    qb, pkb, w = _score_inputs(T, H, D, T // kp, seed=6)
    ops = ora.Operands(qb.reshape(T, H, D), w, pkb)
    full, cond = ora.score_rows_full(ops, None, kp, np.arange(T))
    fin = np.isfinite(full)
    assert np.all(np.abs(full[fin]) <= cond[fin] * (1 + 1e-15))
    opsp = ora.Operands(qb.reshape(T, H, D), np.abs(w), pkb)
    fp, cp = ora.score_rows_full(opsp, None, kp, np.arange(T))
    assert np.array_equal(fp[np.isfinite(fp)], cp[np.isfinite(fp)])


def test_fp8_operands_equal_dequantised_bf16(ora):
    """The FP8 path scores the dequantised values e*s: with codes whose
    dequantised values are exact in bf16 the two paths agree exactly."""
    T, H, D, kp = 32, 2, 128, 4
    gen = torch.Generator().manual_seed(7)
    qc = torch.randint(0, 0x70, (T, H, D), generator=gen).to(torch.uint8).numpy()
    pc = torch.randint(0, 0x70, (T // kp, D), generator=gen).to(torch.uint8).numpy()
    qs = (2.0 ** torch.randint(-4, 4, (T, H), generator=gen).double()).float().numpy()
    ps = (2.0 ** torch.randint(-4, 4, (T // kp,), generator=gen).double()).float().numpy()
    w = (torch.randn(T, H, generator=gen)).numpy()
    deq = lambda c: np.vectorize(ora.e4m3_to_double)(c)
    qv = deq(qc) * qs[..., None]
    pv = deq(pc) * ps[..., None]
    a = ora.score_rows_full(ora.Operands(qc, w, pc, qs, ps), None, kp, np.arange(T))[0]
    b = ora.score_rows_full(ora.Operands(bf16_bits_of(qv.astype(np.float32)), w,
                                         bf16_bits_of(pv.astype(np.float32))),
                            None, kp, np.arange(T))[0]
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# Expansion + tail, prefix visibility, packed THD
# ---------------------------------------------------------------------------

def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, vals = line.split(":")
            rows[key.strip()] = [int(v) for v in vals.split()]
    return rows


def test_expand_golden_worked_example(ora):
    g = _read_golden("expand_kp4_worked.txt")
    kp, Kp = 4, 2
    cu = np.array(g["cu_seqlens"], np.int32)
    rows = np.array(g["rows"], np.int64)
    sel = np.array(g["sel"], np.int32).reshape(len(rows), Kp)
    for tail in (1, 0):
        out = ora.expand_rows(sel, cu, int(cu[-1]), kp, Kp, bool(tail), rows)
        want = np.array(g["out_tail%d" % tail], np.int32).reshape(len(rows), Kp * kp + kp - 1)
        assert np.array_equal(out, want)


@pytest.mark.parametrize("packed", [False, True])
def test_short_prefix_fully_visible(ora, packed):
    """[MG] Testing (test_kpool_causal_tail): every query whose document-local
    prefix fits the budget (tau+1 <= index_topk) sees exactly its full causal
    prefix, packed and unpacked, on a strided subset of queries."""
    wl = W.Workload("t", T=160, H=2, D=16, kpool=4, index_topk=32,
                    n_docs=3 if packed else 1, doc_len_range=(20, 90))
    inp = W.make_inputs(wl)
    cu = inp.cu_seqlens.numpy()
    pk = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(), cu, wl.kpool)
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pk)
    rows = np.arange(0, wl.T, 3)
    out = ora.select_rows(ops, cu, wl.kpool, wl.Kp, rows)
    exp = ora.expand_rows(out["sel"], cu, wl.T, wl.kpool, wl.Kp, True, rows)
    checked = 0
    for i, t in enumerate(rows):
        d = np.searchsorted(cu, t, side="right") - 1
        tau = t - cu[d]
        toks = exp[i][exp[i] >= 0]
        assert np.all(np.diff(toks) > 0)
        assert toks.size == 0 or (toks[0] >= cu[d] and toks[-1] <= t)
        if tau + 1 <= wl.index_topk:
            assert np.array_equal(toks, np.arange(cu[d], t + 1))
            checked += 1
        else:
            assert toks.size == wl.Kp * wl.kpool + (tau + 1) % wl.kpool
    assert checked > 10


def test_packed_equals_per_document(ora):
    """Packed THD selection/expansion = per-document results re-indexed."""
    wl = W.Workload("t", T=300, H=2, D=16, kpool=4, index_topk=16, n_docs=3,
                    doc_len_range=(40, 200))
    inp = W.make_inputs(wl)
    cu = inp.cu_seqlens.numpy()
    kb, gb, qb = W.bits(inp.k), W.bits(inp.gate), W.bits(inp.q)
    w, ape = inp.w.numpy(), inp.ape.numpy()
    pk = ora.compress(kb, gb, ape, cu, 4)
    cp = ora.cu_pools(cu, 4)
    out = ora.select_rows(ora.Operands(qb, w, pk), cu, 4, 4, np.arange(wl.T))
    exp = ora.expand_rows(out["sel"], cu, wl.T, 4, 4, True, np.arange(wl.T))
    for d in range(3):
        a, b = cu[d], cu[d + 1]
        pkd = ora.compress(kb[a:b], gb[a:b], ape, None, 4)
        od = ora.select_rows(ora.Operands(qb[a:b], w[a:b], pkd), None, 4, 4, np.arange(b - a))
        ed = ora.expand_rows(od["sel"], None, b - a, 4, 4, True, np.arange(b - a))
        sel_d = np.where(od["sel"] >= 0, od["sel"] + cp[d], -1)
        assert np.array_equal(out["sel"][a:b], sel_d)
        assert np.array_equal(exp[a:b], np.where(ed >= 0, ed + a, -1))


def test_compress_condition_scale(ora):
    """cond = sum_s alpha_s |k_s| >= |pk_exact|, with equality when all keys
    of a pool share a sign."""
    kb, gb, ape = _rand_inputs(64, 32, 4, seed=8)
    pk, ex, cond = ora.compress(kb, gb, ape, None, 4, want_cond=True)
    assert np.all(cond >= np.abs(ex) * (1 - 1e-15))
    kp_ = kb & 0x7FFF
    _, ex2, cond2 = ora.compress(kp_, gb, ape, None, 4, want_cond=True)
    assert np.allclose(cond2, ex2, rtol=1e-15, atol=0)


# ---------------------------------------------------------------------------
# Queries at given positions (decode / chunked prefill)
# ---------------------------------------------------------------------------

def _thd_case(seed=7):
    wl = W.Workload("at", T=400, H=3, D=16, kpool=4, index_topk=24, n_docs=3,
                    doc_len_range=(60, 200))
    inp = W.make_inputs(wl, seed=seed)
    cu = inp.cu_seqlens.numpy()
    pk = None
    return wl, inp, cu


def test_chunked_prefill_equals_full_prefill_rows(ora):
    """A chunk of query rows [a, b) of each document, given as its own query
    batch at position offset a - doc_start, gets exactly the plain result of
    rows [a, b) (selection, scores and expansion to key-token indices)."""
    wl, inp, cu = _thd_case()
    kb, gb, qb = W.bits(inp.k), W.bits(inp.gate), W.bits(inp.q)
    w = inp.w.numpy()
    pk = ora.compress(kb, gb, inp.ape.numpy(), cu, wl.kpool)
    full = ora.select_rows(ora.Operands(qb, w, pk), cu, wl.kpool, wl.Kp, np.arange(wl.T))
    full_tok = ora.expand_rows(full["sel"], cu, wl.T, wl.kpool, wl.Kp, True, np.arange(wl.T))
    # chunk of each document: its middle third
    rows, cq, qpos = [], [0], []
    for d in range(3):
        L = cu[d + 1] - cu[d]
        a, b = cu[d] + L // 3, cu[d] + 2 * L // 3
        rows.extend(range(a, b))
        cq.append(cq[-1] + (b - a))
        qpos.append(a - cu[d])
    rows = np.array(rows)
    ops_c = ora.Operands(qb[rows], w[rows], pk)
    got = ora.select_rows_at(ops_c, cq, qpos, cu, wl.kpool, wl.Kp, np.arange(len(rows)))
    assert np.array_equal(got["sel"], full["sel"][rows])
    fin = np.isfinite(full["sel_score"][rows])
    assert np.array_equal(got["sel_score"][fin], full["sel_score"][rows][fin])
    tok = ora.expand_rows_at(got["sel"], cq, qpos, cu, wl.kpool, wl.Kp, True,
                             np.arange(len(rows)))
    assert np.array_equal(tok, full_tok[rows])
    sc, cd = ora.score_pairs_at(ops_c, cq, qpos, cu, wl.kpool, [0, 0], [0, cu[-1] // 4])
    assert np.isneginf(sc[1])     # another document's pool is not visible


def test_decode_queries_see_their_document_prefix(ora):
    """One decode query per document at its last position equals the last row
    of the plain result; a position past the keys sees every pool (clamped)."""
    wl, inp, cu = _thd_case(seed=8)
    kb, gb, qb = W.bits(inp.k), W.bits(inp.gate), W.bits(inp.q)
    w = inp.w.numpy()
    pk = ora.compress(kb, gb, inp.ape.numpy(), cu, wl.kpool)
    last = cu[1:] - 1
    full = ora.select_rows(ora.Operands(qb, w, pk), cu, wl.kpool, wl.Kp, last)
    cq = np.arange(4, dtype=np.int32)
    qpos = (cu[1:] - cu[:-1] - 1).astype(np.int32)
    ops_d = ora.Operands(qb[last], w[last], pk)
    got = ora.select_rows_at(ops_d, cq, qpos, cu, wl.kpool, wl.Kp, np.arange(3))
    assert np.array_equal(got["sel"], full["sel"])
    far = ora.select_rows_at(ops_d, cq, qpos + 1000, cu, wl.kpool, 1000, np.arange(3))
    cp = ora.cu_pools(cu, wl.kpool)
    assert list(far["n_sel"]) == list(np.diff(cp))


def _fp8_onehot_cases():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "fp8_onehot_worked.txt")
    cases = []
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        v, j, e, cpos, cneg = line.split()
        cases.append((float(v), int(j), int(e), int(cpos, 16), int(cneg, 16)))
    return cases


def _fp8_onehot_expected(v, j, cpos, cneg):
    signs = np.array([(-1) ** bin(i & j).count("1") for i in range(128)]) * np.sign(v)
    return np.where(signs > 0, cpos, cneg).astype(np.uint8)


def test_fp8_chain_hand_worked_onehot(ora):
    """One-hot rows through the FP8 input path: codes and scales worked out by
    hand (tests/golden/fp8_onehot_worked.txt), including an exact E4M3 tie."""
    cases = _fp8_onehot_cases()
    x = torch.zeros(len(cases), 128, dtype=torch.float32)
    for r, (v, j, _, _, _) in enumerate(cases):
        x[r, j] = v
    codes, scales = ora.fp8_rows(W.bits(x.to(torch.bfloat16)))
    for r, (v, j, e, cpos, cneg) in enumerate(cases):
        assert scales[r] == 2.0 ** e, (v, j, scales[r])
        assert np.array_equal(codes[r], _fp8_onehot_expected(v, j, cpos, cneg)), (v, j)


def score_select_worked(pad_heads=2, pad_dims=2):
    """The hand-worked fixture tests/golden/score_select_worked.txt as bf16
    inputs, optionally zero-padded to more heads (w = 0) and dimensions."""
    path = os.path.join(os.path.dirname(__file__), "golden", "score_select_worked.txt")
    lines = [ln for ln in open(path) if ln.strip() and not ln.startswith("#")]
    kv = [float(x) for x in lines[0].split(":")[1].split()]
    k = torch.zeros(5, pad_dims)
    k[:, :2] = torch.tensor(kv).view(5, 2)
    q = torch.zeros(5, pad_heads, pad_dims)
    q[:, 0, 0] = 1.0
    q[:, 1, 1] = 2.0
    w = torch.zeros(5, pad_heads)
    w[:, 0] = 1.0
    w[:, 1] = -0.5
    want_idx, want_sc = [], []
    for ln in lines[1:]:
        idx, sc = ln.split(":")[1].split("|")
        want_idx.append([int(x) for x in idx.split()])
        want_sc.append([float(x) for x in sc.split()])
    return (q.to(torch.bfloat16), k.to(torch.bfloat16), w, np.array(want_idx, np.int32),
            np.array(want_sc, np.float64))


def test_score_and_selection_hand_worked(ora):
    q, k, w, want_idx, want_sc = score_select_worked()
    ops = ora.Operands(W.bits(q), w.numpy(), W.bits(k))
    o = ora.select_rows(ops, None, 1, 2, np.arange(5))
    assert np.array_equal(o["sel"], want_idx)
    got = np.where(want_idx >= 0, o["sel_score"], -np.inf)
    assert np.array_equal(got, want_sc)


def compress_worked_cases():
    """tests/golden/compress_worked.txt: one hand-worked pool per line (kpool,
    gate and keys per slot, ape = float32(ln m + c) per slot, the pooled key)."""
    cases = []
    for line in open(os.path.join(GOLDEN, "compress_worked.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        f = [x.split() for x in line.split("|")]
        kp = int(f[0][0])
        gate, m, c, keys = ([float(v) for v in f[i]] for i in range(1, 5))
        assert len(gate) == len(m) == len(c) == len(keys) == kp
        cases.append((kp, gate, m, c, keys, float(f[5][0])))
    return cases


def compress_worked_inputs(kp, D=32):
    """The fixture's cases of one kpool laid out as one pool of D dimensions,
    case i in dimension i, zeros elsewhere (whose pooled key is 0).  Returns
    bf16 k and gate [kp, D] (torch), ape [kp, D] float32 and the expected
    pooled keys [D] (float64)."""
    cases = [cs for cs in compress_worked_cases() if cs[0] == kp]
    assert 0 < len(cases) <= D
    k = torch.zeros(kp, D)
    gate = torch.zeros(kp, D)
    ape = np.zeros((kp, D), np.float32)
    want = np.zeros(D)
    for d, (_, g, m, c, keys, pk) in enumerate(cases):
        for s in range(kp):
            k[s, d] = keys[s]
            gate[s, d] = g[s]
            ape[s, d] = np.float32(math.log(m[s]) + c[s])
        want[d] = pk
    kb, gb = k.to(torch.bfloat16), gate.to(torch.bfloat16)
    assert torch.equal(kb.float(), k) and torch.equal(gb.float(), gate)   # BF16-exact inputs
    return kb, gb, ape, want


@pytest.mark.parametrize("kp", [2, 3, 4])
def test_compress_hand_worked_moderate_logits(ora, kp):
    """Hand-worked pooled keys at moderate logits (tests/golden/compress_worked.txt):
    softmax weights that are small rationals (1/4, 3/4, 1/8, 0.1 .. 0.4), so a
    softmax at another temperature, of the negated logits, over reversed slots,
    or without the gate or the ape term gives another pooled key."""
    kb, gb, ape, want = compress_worked_inputs(kp)
    pk = ora.compress(W.bits(kb), W.bits(gb), ape, None, kp)
    assert pk.shape == (1, 32)
    assert np.array_equal(bf16_val(pk[0]), want), (bf16_val(pk[0]), want)


# ---------------------------------------------------------------------------
# The key path in front of compression (linear_wk -> k_norm, gate projection)
# ---------------------------------------------------------------------------

def _nearest_bf16(bits, exact):
    """Each BF16 value is within half a BF16 spacing of its exact value (8
    significant bits: spacing 2^(floor(log2|v|) - 7))."""
    v = bf16_val(bits)
    nz = exact != 0
    e = np.floor(np.log2(np.abs(np.where(nz, exact, 1.0))))
    half = 2.0 ** (e - 8)
    return bool(np.all(np.abs(v - exact)[nz] <= half[nz]) and np.all(v[~nz] == 0))


def _proj_inputs(T=24, hidden=96, D=32, seed=12):
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(T, hidden, generator=gen).to(torch.bfloat16)
    w = (torch.randn(2 * D, hidden, generator=gen) / math.sqrt(hidden)).to(torch.bfloat16)
    gamma = (1.0 + 0.1 * torch.randn(D, generator=gen)).float()
    beta = (0.1 * torch.randn(D, generator=gen)).float()
    return x, w, gamma, beta


def test_project_keys_is_a_matmul_then_layer_norm(ora):
    """The projections equal numpy's float64 matmul of the BF16 operands (the
    first D weight rows give the keys, the next D the gate), and the key
    normalisation equals torch's float64 layer_norm (biased variance, eps
    inside the square root, weight and bias) of the BF16-rounded projection."""
    x, w, gamma, beta = _proj_inputs()
    eps = 1e-6
    k, g, kp_ex, k_ex, g_ex, k_cond = ora.project_keys(W.bits(x), W.bits(w), gamma.numpy(),
                                                       beta.numpy(), eps, want_exact=True)
    assert np.all(k_cond >= np.abs(k_ex) * (1 - 1e-12))   # the scale bounds the value
    xd, wd = x.double().numpy(), w.double().numpy()
    D = w.shape[0] // 2
    assert np.allclose(kp_ex, xd @ wd[:D].T, rtol=1e-12, atol=1e-13)
    assert np.allclose(g_ex, xd @ wd[D:].T, rtol=1e-12, atol=1e-13)
    assert _nearest_bf16(g, g_ex)
    kp_r = bf16_val(bf16_bits_of(kp_ex.astype(np.float32)))
    ln = torch.nn.functional.layer_norm(torch.from_numpy(kp_r), (D,),
                                        gamma.double(), beta.double(), eps).numpy()
    assert np.allclose(k_ex, ln, rtol=1e-10, atol=1e-12)
    assert _nearest_bf16(k, k_ex)


def test_project_keys_closed_forms(ora):
    """A zero input row normalises to the bias exactly; a projection that takes
    only the values +a and -a in equal numbers normalises to
    +-a / sqrt(a^2 + eps) * gamma + beta."""
    T, hidden, D = 3, 64, 32
    x = torch.zeros(T, hidden)
    x[1, 0] = 1.0
    x[2, 0] = 0.5
    w = torch.zeros(2 * D, hidden)
    w[:D, 0] = torch.tensor([2.0, -2.0] * (D // 2))      # kproj = +-2 x[:, 0]
    w[D:, 1] = 1.0
    gamma = torch.linspace(0.5, 1.5, D)
    beta = torch.linspace(-0.25, 0.25, D)
    eps = 1e-6
    k, g, _, k_ex, _, _ = ora.project_keys(W.bits(x.to(torch.bfloat16)),
                                           W.bits(w.to(torch.bfloat16)), gamma.numpy(),
                                           beta.numpy(), eps, want_exact=True)
    assert np.array_equal(k_ex[0], beta.double().numpy())
    for t, a in ((1, 2.0), (2, 1.0)):
        sign = np.array([1.0, -1.0] * (D // 2))
        want = sign * a / math.sqrt(a * a + eps) * gamma.double().numpy() + beta.double().numpy()
        assert np.allclose(k_ex[t], want, rtol=1e-14, atol=1e-15)
    assert not np.any(bf16_val(g))     # the gate column of x is zero



# ---------------------------------------------------------------------------
# The sparse attention that consumes the selection (absorbed NoPE form)
# ---------------------------------------------------------------------------

def _frac(x: str) -> float:
    if "/" in x:
        a, b = x.split("/")
        return float(a) / float(b)
    return float(x)


def _ln(x: str) -> float:
    x = x.strip()
    if x == "-inf":
        return -math.inf
    assert x.startswith("ln ")
    return math.log(_frac(x[3:]))


def sparse_attn_worked():
    """tests/golden/sparse_attn_worked.txt: the token table {j: (c0, c1)} and
    the cases (scale, q0, indices, o0, o1, lse)."""
    table, cases = {}, []
    for line in open(os.path.join(GOLDEN, "sparse_attn_worked.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = [x.strip() for x in line.split("|")]
        if f[0] == "token":
            table[int(f[1])] = (_frac(f[2]), _frac(f[3]))
        else:
            assert f[0] == "case"
            cases.append((_ln(f[1]), _frac(f[2]), [int(v) for v in f[3].split()],
                          _frac(f[4]), _frac(f[5]), _ln(f[6])))
    return table, cases


def sparse_attn_worked_inputs(q0, idx, table, H=2, Dc=8, Tq=1):
    """BF16 q [Tq, H, Dc] with q[:, :, 0] = q0, latent rows [len(table), Dc]
    with dims 0 and 1 from the table, and the index row padded to itself."""
    c = torch.zeros(len(table), Dc)
    for j, (a, v) in table.items():
        c[j, 0], c[j, 1] = a, v
    q = torch.zeros(Tq, H, Dc)
    q[:, :, 0] = q0
    return q.to(torch.bfloat16), c.to(torch.bfloat16), np.array([idx], np.int32)


def test_sparse_attn_hand_worked(ora):
    """Hand-worked weights at moderate scores (tests/golden/sparse_attn_worked.txt)."""
    table, cases = sparse_attn_worked()
    assert len(cases) == 6
    for scale, q0, idx, o0, o1, lse in cases:
        q, c, tok = sparse_attn_worked_inputs(q0, idx, table)
        o, l = ora.sparse_attn(W.bits(q), W.bits(c), tok, scale, np.array([0]))
        want = np.zeros((2, 8))
        want[:, 0], want[:, 1] = o0, o1
        assert np.allclose(o[0], want, rtol=1e-13, atol=1e-14), (idx, o[0, 0, :2])
        if math.isinf(lse):
            assert np.all(np.isneginf(l[0]))
        else:
            assert np.allclose(l[0], lse, rtol=1e-13, atol=1e-14)


def _attn_inputs(T=40, H=3, Dc=16, seed=21):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(T, H, Dc, generator=gen).to(torch.bfloat16)
    c = torch.randn(T, Dc, generator=gen).to(torch.bfloat16)
    return q, c


def test_sparse_attn_matches_scipy_softmax(ora):
    """Against scipy's softmax and logsumexp of numpy's float64 scores, on
    random token subsets with -1 padding (the softmax runs over the tokens of
    each head separately)."""
    from scipy.special import logsumexp, softmax
    q, c = _attn_inputs()
    qd, cd = q.double().numpy(), c.double().numpy()
    rng = np.random.default_rng(3)
    rows = np.array([5, 17, 39])
    Wd = 12
    tok = np.full((3, Wd), -1, np.int32)
    for i, t in enumerate(rows):
        sel = np.sort(rng.choice(t + 1, size=min(t + 1, 9), replace=False))
        tok[i, :len(sel)] = sel
    scale = 0.3
    o, lse = ora.sparse_attn(W.bits(q), W.bits(c), tok, scale, rows)
    for i, t in enumerate(rows):
        sel = tok[i][tok[i] >= 0]
        s = scale * qd[t] @ cd[sel].T                      # [H, n]
        assert np.allclose(lse[i], logsumexp(s, axis=1), rtol=1e-13, atol=1e-13)
        assert np.allclose(o[i], softmax(s, axis=1) @ cd[sel], rtol=1e-12, atol=1e-13)


def test_sparse_attn_closed_forms(ora):
    """One token: o is that token's latent row and lse its score; tokens with
    identical latent rows: o is the row and lse = s + log(n); an order change
    of the token list changes nothing; an empty row gives o = 0, lse = -inf."""
    q, c = _attn_inputs(T=16, H=2, Dc=8)
    qd, cd = q.double().numpy(), c.double().numpy()
    tok = np.array([[7, -1, -1, -1], [-1, -1, -1, -1], [3, 9, 1, -1], [9, 1, -1, 3]], np.int32)
    rows = np.array([10, 11, 12, 12])
    o, lse = ora.sparse_attn(W.bits(q), W.bits(c), tok, 0.5, rows)
    assert np.array_equal(o[0], np.tile(cd[7], (2, 1)))
    assert np.allclose(lse[0], 0.5 * qd[10] @ cd[7], rtol=1e-15, atol=1e-15)
    assert np.all(o[1] == 0) and np.all(np.isneginf(lse[1]))
    assert np.allclose(o[2], o[3], rtol=1e-14, atol=1e-15) and np.allclose(lse[2], lse[3])
    c_same = c.clone()
    c_same[[1, 3, 9]] = c[4]
    o2, lse2 = ora.sparse_attn(W.bits(q), W.bits(c_same), tok[2:3], 0.5, rows[2:3])
    assert np.allclose(o2[0], np.tile(cd[4], (2, 1)), rtol=1e-14, atol=1e-15)
    assert np.allclose(lse2[0], 0.5 * qd[12] @ cd[4] + math.log(3), rtol=1e-14)
