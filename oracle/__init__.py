"""Plain CPU oracle for the KPool DSA indexer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its binding) never imports it.

The arithmetic lives in ``kpool_oracle.c`` (plain C, double precision, its
own BF16/E4M3 rounding, an explicit Hadamard matrix, full-sort selection).
This module only compiles that file with gcc and marshals numpy arrays.

What each function follows (page titles and sections):

* ``compress`` -- Megatron-LM PR "GLM5.3 Flash (KDA + mHC + KPool DSA)
  support + FP8", Changes section 3 (per-dimension softmax over slots,
  FP32 accumulation, one BF16 rounding) and SkyRL PR "GLM-5.3-Flash
  (glm5_next) Megatron support", commit "k-pool indexer"
  (``gate_score + ape`` softmax, per-segment pools).
* ``fp8_rows`` -- the same Megatron-LM section 3 (FP32 Hadamard -> BF16 ->
  E4M3 with a power-of-two row scale) and its Testing section (the
  Hadamard-matrix reference).
* ``select_rows`` / ``score_pairs`` / ``score_rows_full`` -- pool scoring
  ``sum_h w * relu(q . pk)`` over complete causal pools and top
  ``index_topk // kpool`` selection, ties to the lower pool index.
* ``expand_rows`` -- expansion of pools to tokens plus the causal tail
  (``always_select_tail``).
* ``sparse_attn`` -- the sparse attention that consumes the selection:
  xtuner PR "GLM-5.3-Flash F5: NoPE DSA + KPool indexer + clamped
  SwiGLU", Summary (NoPE sparse attention, a FlashMLA-style SparseMLA
  forward over the selected tokens) and Megatron-LM PR Changes section 3
  ("NoPE": no positional slice in the absorbed query); in the absorbed
  form the latent rows are both keys and values.
* ``project_keys`` -- the key path in front of compression: Megatron-LM PR
  Changes section 4 (linear_wk and k_norm in BF16, unquantized) and section
  3 / SkyRL commit "k-pool indexer" (the BF16 compression gate); k_norm is
  read as a LayerNorm with weight and bias.

Every function is pinned by ``tests/test_oracle_pins.py``; none is left
unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kpool_oracle.c")
_LIB = os.path.join(_HERE, "libkpool_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over query rows).  Idempotent."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        sig = {
            "ora_bf16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
            "ora_bf16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
            "ora_e4m3_to_double": (ctypes.c_double, [ctypes.c_uint8]),
            "ora_e4m3_from_double": (ctypes.c_uint8, [ctypes.c_double]),
            "ora_pow2_scale": (ctypes.c_double, [ctypes.c_double]),
            "ora_cu_pools": (i64, [P, i32, i32, P]),
            "ora_compress": (None, [P, P, P, P, i32, i32, i32, P, P, P]),
            "ora_pool_weights": (None, [P, P, i64, i32, i32, P]),
            "ora_project_keys": (None, [P, P, P, P, ctypes.c_double, i64, i32, i32, P, P, P, P,
                                        P, P]),
            "ora_hadamard_matrix": (None, [i32, P]),
            "ora_fp8_rows": (None, [P, i64, i32, P, P, P, P]),
            "ora_score_pairs": (None, [P, P, P, P, P, i32, P, i32, i32, i32, i32, i64,
                                       P, P, i64, P, P]),
            "ora_select_rows": (None, [P, P, P, P, P, i32, P, i32, i32, i32, i32, i64, i32,
                                       P, i64, P, P, P, P, P]),
            "ora_score_rows_full": (None, [P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                           i64, P, i64, P, P]),
            "ora_expand_rows": (None, [P, P, i32, i32, i32, i32, P, i64, P]),
            "ora_score_pairs_at": (None, [P, P, P, P, P, i32, P, P, P, i32, i32, i32, i32, i64,
                                          P, P, i64, P, P]),
            "ora_select_rows_at": (None, [P, P, P, P, P, i32, P, P, P, i32, i32, i32, i32, i64,
                                          i32, P, i64, P, P, P, P, P]),
            "ora_expand_rows_at": (None, [P, P, P, P, i32, i32, i32, i32, P, i64, P]),
            "ora_num_threads": (i32, []),
            "ora_sparse_attn": (None, [P, P, P, i32, i32, i32, ctypes.c_double, P, i64, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _seqlens(cu_seqlens, T):
    if cu_seqlens is None:
        return np.array([0, T], dtype=np.int32)
    return _c(cu_seqlens, np.int32)


# -- formats -----------------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return _load().ora_bf16_to_double(int(bits))


def bf16_from_double(x: float) -> int:
    return int(_load().ora_bf16_from_double(float(x)))


def e4m3_to_double(code: int) -> float:
    return _load().ora_e4m3_to_double(int(code))


def e4m3_from_double(x: float) -> int:
    return int(_load().ora_e4m3_from_double(float(x)))


def pow2_scale(amax: float) -> float:
    return _load().ora_pow2_scale(float(amax))


def hadamard_matrix(n: int) -> np.ndarray:
    out = np.empty((n, n), dtype=np.float64)
    _load().ora_hadamard_matrix(n, _ptr(out))
    return out


def num_threads() -> int:
    return int(_load().ora_num_threads())


# -- method ------------------------------------------------------------------

def cu_pools(cu_seqlens, kp: int) -> np.ndarray:
    cs = _c(cu_seqlens, np.int32)
    out = np.empty(len(cs), dtype=np.int32)
    _load().ora_cu_pools(_ptr(cs), len(cs) - 1, kp, _ptr(out))
    return out


def compress(k_bits, gate_bits, ape, cu_seqlens, kp: int, want_exact: bool = False,
             want_cond: bool = False):
    """k_bits, gate_bits: uint16 bf16 bit patterns [T, D]; ape float32 [kp, D].
    Returns pk bits uint16 [P_total, D]; with want_exact also the unrounded
    doubles, with want_cond also the condition scale sum_s alpha_s |k_s|."""
    k_bits = _c(k_bits, np.uint16)
    gate_bits = _c(gate_bits, np.uint16)
    ape = _c(ape, np.float32)
    T, D = k_bits.shape
    cs = _seqlens(cu_seqlens, T)
    P = int(cu_pools(cs, kp)[-1])
    pk = np.zeros((P, D), dtype=np.uint16)
    exact = np.zeros((P, D), dtype=np.float64) if (want_exact or want_cond) else None
    cond = np.zeros((P, D), dtype=np.float64) if want_cond else None
    _load().ora_compress(_ptr(k_bits), _ptr(gate_bits), _ptr(ape), _ptr(cs), len(cs) - 1,
                         D, kp, _ptr(pk), _ptr(exact), _ptr(cond))
    if want_cond:
        return pk, exact, cond
    return (pk, exact) if want_exact else pk


def project_keys(x_bits, w_bits, gamma, beta, eps: float, want_exact: bool = False):
    """The key path in front of compression: x_bits bf16 [T, hidden], w_bits
    bf16 [2D, hidden] (W_k rows then the gate projection's rows), gamma and
    beta float32 [D].  Returns (k bits, gate bits) uint16 [T, D]; with
    want_exact also the unrounded (kproj, k, gate) doubles and the condition
    scale of each normalised key."""
    x_bits = _c(x_bits, np.uint16)
    w_bits = _c(w_bits, np.uint16)
    gamma = _c(gamma, np.float32)
    beta = _c(beta, np.float32)
    T, hidden = x_bits.shape
    D = w_bits.shape[0] // 2
    assert w_bits.shape == (2 * D, hidden) and D <= 256 and gamma.shape == beta.shape == (D,)
    k = np.empty((T, D), np.uint16)
    g = np.empty((T, D), np.uint16)
    ex = [np.empty((T, D), np.float64) for _ in range(4)] if want_exact else [None] * 4
    _load().ora_project_keys(_ptr(x_bits), _ptr(w_bits), _ptr(gamma), _ptr(beta), float(eps), T,
                             hidden, D, _ptr(k), _ptr(g), _ptr(ex[0]), _ptr(ex[1]), _ptr(ex[2]),
                             _ptr(ex[3]))
    return (k, g, ex[0], ex[1], ex[2], ex[3]) if want_exact else (k, g)


def pool_weights(gate_bits, ape, first_token: int, kp: int) -> np.ndarray:
    gate_bits = _c(gate_bits, np.uint16)
    ape = _c(ape, np.float32)
    D = gate_bits.shape[1]
    out = np.empty((kp, D), dtype=np.float64)
    _load().ora_pool_weights(_ptr(gate_bits), _ptr(ape), first_token, D, kp, _ptr(out))
    return out


def fp8_rows(x_bits, want_intermediate: bool = False):
    """x_bits: uint16 bf16 [rows, D].  Returns (codes uint8 [rows, D],
    scales float32 [rows]) and optionally (y double, b bf16 bits)."""
    x_bits = _c(x_bits, np.uint16)
    rows, D = x_bits.reshape(-1, x_bits.shape[-1]).shape
    codes = np.empty((rows, D), dtype=np.uint8)
    scales = np.empty(rows, dtype=np.float32)
    y = np.empty((rows, D), dtype=np.float64) if want_intermediate else None
    b = np.empty((rows, D), dtype=np.uint16) if want_intermediate else None
    _load().ora_fp8_rows(_ptr(x_bits), rows, D, _ptr(codes), _ptr(scales), _ptr(y), _ptr(b))
    if want_intermediate:
        return codes, scales, y, b
    return codes, scales


class Operands:
    """Scoring operands: bf16 (q, pk as uint16 bits) or FP8 (uint8 codes plus
    float32 scales).  q is [T, H, D], w [T, H], pk [P, D]."""

    def __init__(self, q, w, pk, q_scale=None, pk_scale=None):
        self.fp8 = q_scale is not None
        if self.fp8:
            self.q = _c(q, np.uint8)
            self.pk = _c(pk, np.uint8)
            self.qs = _c(q_scale, np.float32)
            self.pks = _c(pk_scale, np.float32)
        else:
            self.q = _c(q, np.uint16)
            self.pk = _c(pk, np.uint16)
            self.qs = None
            self.pks = None
        self.w = _c(w, np.float32)
        self.T, self.H, self.D = self.q.shape
        self.P = self.pk.shape[0]

    def args(self):
        return (_ptr(self.q), _ptr(self.qs), _ptr(self.w), _ptr(self.pk), _ptr(self.pks),
                int(self.fp8))


def select_rows(ops: Operands, cu_seqlens, kp: int, Kp: int, rows):
    cs = _seqlens(cu_seqlens, ops.T)
    rows = _c(rows, np.int64)
    n = len(rows)
    sel = np.empty((n, Kp), dtype=np.int32)
    sel_score = np.empty((n, Kp), dtype=np.float64)
    kth = np.empty(n, dtype=np.float64)
    kth_cond = np.empty(n, dtype=np.float64)
    n_sel = np.empty(n, dtype=np.int32)
    _load().ora_select_rows(*ops.args(), _ptr(cs), len(cs) - 1, ops.H, ops.D, kp, ops.P, Kp,
                            _ptr(rows), n, _ptr(sel), _ptr(sel_score), _ptr(kth),
                            _ptr(kth_cond), _ptr(n_sel))
    return dict(sel=sel, sel_score=sel_score, kth=kth, kth_cond=kth_cond, n_sel=n_sel)


def score_pairs(ops: Operands, cu_seqlens, kp: int, rows, pools):
    cs = _seqlens(cu_seqlens, ops.T)
    rows = _c(rows, np.int64)
    pools = _c(pools, np.int64)
    n = len(rows)
    sc = np.empty(n, dtype=np.float64)
    cd = np.empty(n, dtype=np.float64)
    _load().ora_score_pairs(*ops.args(), _ptr(cs), len(cs) - 1, ops.H, ops.D, kp, ops.P,
                            _ptr(rows), _ptr(pools), n, _ptr(sc), _ptr(cd))
    return sc, cd


def score_rows_full(ops: Operands, cu_seqlens, kp: int, rows):
    cs = _seqlens(cu_seqlens, ops.T)
    rows = _c(rows, np.int64)
    n = len(rows)
    out = np.empty((n, ops.P), dtype=np.float64)
    cond = np.empty((n, ops.P), dtype=np.float64)
    _load().ora_score_rows_full(*ops.args(), _ptr(cs), len(cs) - 1, ops.H, ops.D, kp,
                                ops.P, _ptr(rows), n, _ptr(out), _ptr(cond))
    return out, cond


def expand_rows(sel, cu_seqlens, T: int, kp: int, Kp: int, tail: bool, rows):
    cs = _seqlens(cu_seqlens, T)
    rows = _c(rows, np.int64)
    sel = _c(sel, np.int32)
    n = len(rows)
    W = Kp * kp + kp - 1
    out = np.empty((n, W), dtype=np.int32)
    _load().ora_expand_rows(_ptr(sel), _ptr(cs), len(cs) - 1, kp, Kp, int(bool(tail)),
                            _ptr(rows), n, _ptr(out))
    return out


# -- queries at given positions (decode / chunked prefill) --------------------
# Document d's query rows are [cu_q[d], cu_q[d+1]) of q (and w); its i-th query
# sits at document-local position q_pos[d] + i of a key sequence whose tokens
# are [cu_k[d], cu_k[d+1]) (pooled keys: floor(L_k / kpool) per document).

def select_rows_at(ops: Operands, cu_q, q_pos, cu_k, kp: int, Kp: int, rows):
    cq, qp, ck = _c(cu_q, np.int32), _c(q_pos, np.int32), _c(cu_k, np.int32)
    rows = _c(rows, np.int64)
    n = len(rows)
    sel = np.empty((n, Kp), dtype=np.int32)
    sel_score = np.empty((n, Kp), dtype=np.float64)
    kth = np.empty(n, dtype=np.float64)
    kth_cond = np.empty(n, dtype=np.float64)
    n_sel = np.empty(n, dtype=np.int32)
    _load().ora_select_rows_at(*ops.args(), _ptr(cq), _ptr(qp), _ptr(ck), len(cq) - 1, ops.H,
                               ops.D, kp, ops.P, Kp, _ptr(rows), n, _ptr(sel), _ptr(sel_score),
                               _ptr(kth), _ptr(kth_cond), _ptr(n_sel))
    return dict(sel=sel, sel_score=sel_score, kth=kth, kth_cond=kth_cond, n_sel=n_sel)


def score_pairs_at(ops: Operands, cu_q, q_pos, cu_k, kp: int, rows, pools):
    cq, qp, ck = _c(cu_q, np.int32), _c(q_pos, np.int32), _c(cu_k, np.int32)
    rows = _c(rows, np.int64)
    pools = _c(pools, np.int64)
    n = len(rows)
    sc = np.empty(n, dtype=np.float64)
    cd = np.empty(n, dtype=np.float64)
    _load().ora_score_pairs_at(*ops.args(), _ptr(cq), _ptr(qp), _ptr(ck), len(cq) - 1, ops.H,
                               ops.D, kp, ops.P, _ptr(rows), _ptr(pools), n, _ptr(sc), _ptr(cd))
    return sc, cd


def expand_rows_at(sel, cu_q, q_pos, cu_k, kp: int, Kp: int, tail: bool, rows):
    cq, qp, ck = _c(cu_q, np.int32), _c(q_pos, np.int32), _c(cu_k, np.int32)
    rows = _c(rows, np.int64)
    sel = _c(sel, np.int32)
    n = len(rows)
    W = Kp * kp + kp - 1
    out = np.empty((n, W), dtype=np.int32)
    _load().ora_expand_rows_at(_ptr(sel), _ptr(cq), _ptr(qp), _ptr(ck), len(cq) - 1, kp, Kp,
                               int(bool(tail)), _ptr(rows), n, _ptr(out))
    return out


def sparse_attn(q_bits, c_bits, tok, scale: float, rows):
    """Sparse attention over the selected tokens (absorbed NoPE form: keys and
    values are the latent rows c).  q_bits bf16 bits [T, H, Dc], c_bits bf16
    bits [Tk, Dc], tok int32 [len(rows), W] token indices (-1 = none) for the
    query rows `rows`.  Returns (o float64 [len(rows), H, Dc], lse float64
    [len(rows), H]); lse is the natural-log sum of exp of the scaled scores."""
    q_bits = _c(q_bits, np.uint16)
    c_bits = _c(c_bits, np.uint16)
    tok = _c(tok, np.int32)
    rows = _c(rows, np.int64)
    T, H, Dc = q_bits.shape
    n, W = tok.shape
    assert n == len(rows) and c_bits.shape[1] == Dc
    o = np.empty((n, H, Dc), np.float64)
    lse = np.empty((n, H), np.float64)
    _load().ora_sparse_attn(_ptr(q_bits), _ptr(c_bits), _ptr(tok), W, H, Dc, float(scale),
                            _ptr(rows), n, _ptr(o), _ptr(lse))
    return o, lse
