"""Parity comparison helpers shared by the GPU tests (test infrastructure).

Tolerances (the stated bars for this path):
  * pooled keys: at most 1 BF16 ulp apart (distance of ordered bit patterns);
  * scores: |gpu - oracle| <= tol * S, S = sum_h |w| relu(q . pk) the score's
    condition scale (w has random sign, so the score itself can cancel to
    ~0), tol = 1e-3 with FP32 accumulation, 5e-2 in FP8 mode end to end;
  * selections: equal sets except for swaps among pools whose oracle scores
    lie within tol * (S_x + S_max) of the oracle's Kp-th score;
  * expansion / tail: bit-exact.
"""
import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def ordered_bf16(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(ordered_bf16(a) - ordered_bf16(b))


def check_pooled_keys(got_bits, want_bits, exact, cond, name=""):
    """Pooled keys: at most 1 BF16 ulp from the oracle's correctly rounded
    value.  Where the weighted sum cancels (|exact| far below its condition
    scale sum_s alpha_s |k_s|), FP32 evaluation -- the precision the method
    prescribes -- carries an absolute error of a few 2^-24 * cond that can
    exceed an ulp of the tiny result; there the allowance is
    |gpu - exact| <= 2^-20 * cond.  Returns the number of such elements."""
    assert got_bits.shape == want_bits.shape
    dist = bf16_ulp_distance(got_bits, want_bits)
    over = dist > 1
    if over.any():
        got = (got_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        err = np.abs(got[over] - exact[over])
        ok = err <= 2.0 ** -20 * cond[over]
        assert ok.all(), "%s: %d pooled-key elements beyond 1 ulp and the FP32 allowance" % (
            name, int((~ok).sum()))
        assert over.mean() < 1e-4, "%s: too many cancellation cases (%d)" % (name, int(over.sum()))
    return int(over.sum())


def check_selection(ora, ops, cu_seqlens, kp, Kp, rows, gpu_idx, gpu_score, tol, name=""):
    """rows: int64 array of query rows; gpu_idx/gpu_score: [len(rows), Kp]
    numpy arrays of the GPU output for those rows (gpu_score None: a path that
    returns only indices; the set checks still run).  Returns a dict of stats;
    raises AssertionError on a violation."""
    rows = np.asarray(rows, dtype=np.int64)
    o = ora.select_rows(ops, cu_seqlens, kp, Kp, rows)
    n_swaps = 0
    pair_r, pair_p = [], []
    for i in range(len(rows)):
        g = gpu_idx[i]
        ns = int(o["n_sel"][i])
        gv = g[g >= 0]
        assert gv.size == ns, "%s row %d: %d selected, oracle %d" % (name, rows[i], gv.size, ns)
        assert np.all(g[ns:] == -1), "%s row %d: padding" % (name, rows[i])
        assert np.all(np.diff(gv) > 0), "%s row %d: not strictly ascending" % (name, rows[i])
        if gpu_score is not None:
            assert np.all(np.isneginf(gpu_score[i][ns:])), "%s row %d: score padding" % (
                name, rows[i])
        pair_r.extend([rows[i]] * ns)
        pair_p.extend(gv.tolist())
        ov = o["sel"][i][: ns]
        if not np.array_equal(gv, ov):
            delta = np.setxor1d(gv, ov)
            pair_r.extend([rows[i]] * delta.size)
            pair_p.extend(delta.tolist())
    sc, cd = ora.score_pairs(ops, cu_seqlens, kp, np.array(pair_r, np.int64),
                             np.array(pair_p, np.int64)) if pair_r else (np.zeros(0), np.zeros(0))
    lut = {}
    for r, p, s, c in zip(pair_r, pair_p, sc, cd):
        lut[(int(r), int(p))] = (s, c)
    max_rel = 0.0
    for i in range(len(rows)):
        r = int(rows[i])
        ns = int(o["n_sel"][i])
        g = gpu_idx[i][:ns]
        for j, p in enumerate(g):
            s, c = lut[(r, int(p))]
            assert np.isfinite(s), "%s row %d: pool %d not causal" % (name, r, p)
            if gpu_score is None:
                continue
            err = abs(float(gpu_score[i][j]) - s)
            lim = tol * c + 1e-30
            max_rel = max(max_rel, err / (c + 1e-30))
            assert err <= lim, "%s row %d pool %d: score %r vs oracle %r (S=%r)" % (
                name, r, p, float(gpu_score[i][j]), s, c)
        ov = o["sel"][i][: ns]
        if not np.array_equal(g, ov):
            delta = np.setxor1d(g, ov)
            n_swaps += delta.size // 2
            kth = o["kth"][i]
            smax = max(lut[(r, int(p))][1] for p in delta)
            for p in delta:
                s, c = lut[(r, int(p))]
                assert abs(s - kth) <= tol * (c + smax), (
                    "%s row %d: pool %d swapped (oracle %r, k-th %r, S %r)" % (name, r, p, s, kth, c))
    return {"rows": len(rows), "swaps": n_swaps, "max_rel_score_err": max_rel}


def check_dense_scores(gpu, ora_scores, ora_cond, tol, name=""):
    fin = np.isfinite(ora_scores)
    assert np.array_equal(np.isfinite(gpu), fin), "%s: causal mask differs" % name
    assert np.all(np.isneginf(gpu[~fin]))
    err = np.abs(gpu[fin].astype(np.float64) - ora_scores[fin])
    lim = tol * ora_cond[fin]
    bad = err > lim
    assert not bad.any(), "%s: %d scores out of tolerance, worst %r" % (
        name, int(bad.sum()), float((err / (ora_cond[fin] + 1e-30)).max()))
    return float((err / (ora_cond[fin] + 1e-30)).max()) if err.size else 0.0


def pools_from_tokens(tok, rows, cu_seqlens, T, kp, n_sel):
    """Recover each row's pool list from its token row (the first n_sel * kp
    entries are whole pools in ascending order): [len(rows), max n_sel]
    global pool indices, -1 padded.  Checks that every group of kp tokens is
    one aligned pool of the row's document."""
    cu = np.asarray(cu_seqlens if cu_seqlens is not None else [0, T], np.int64)
    cp = np.concatenate([[0], np.cumsum((cu[1:] - cu[:-1]) // kp)])
    width = int(max(n_sel)) if len(n_sel) else 0
    out = np.full((len(rows), max(width, 1)), -1, np.int64)
    for i, t in enumerate(rows):
        d = int(np.searchsorted(cu, t, side="right") - 1)
        ns = int(n_sel[i])
        grp = tok[i][: ns * kp].astype(np.int64).reshape(ns, kp) - cu[d]
        assert np.all(grp[:, 0] % kp == 0) and np.all(grp - grp[:, :1] == np.arange(kp)), t
        out[i, :ns] = cp[d] + grp[:, 0] // kp
    return out
