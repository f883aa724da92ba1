"""Per-phase cycle breakdown of the scoring kernel (diagnostics).

Builds the ``phase_timers`` variant of the library (``-DKPOOL_PHASE_TIMERS``:
the same kernels plus clock64 counters around each wait and work phase),
runs ``kpool_score_topk`` on random bf16 inputs of the requested size and
prints, per role (epilogue warps, MMA thread, TMA producer thread), the share
of cycles in each phase, summed over all CTAs.

    python -m sparse_attention_kpool_compress_gb300.phase_report [T ...]
    python -m sparse_attention_kpool_compress_gb300.phase_report decode:B:LO:HI
    python -m sparse_attention_kpool_compress_gb300.phase_report fp8:T

``decode:B:LO:HI`` runs ``kpool_score_topk_at`` on B documents with seeded
key lengths uniform in [LO, HI) and one query each at its last key, with a
workspace that enables the split-pool schedule.
"""
from __future__ import annotations

import ctypes
import json
import sys

import torch

from . import build as B

EPI = ["wait_tile", "loop_overhead", "wait_tmem_full", "tmem_ld_and_math", "append",
       "capacity_check_and_compaction", "final_select_and_store", "other"]
MMA = ["wait_tile", "wait_q_full", "wait_tmem_empty", "wait_pk_full", "issue", "other"]
PROD = ["wait_tile_slot", "wait_q_empty", "wait_pk_empty", "issue", "other"]


def _lib():
    lib = ctypes.CDLL(B.build(variant="phase_timers"))
    P = ctypes.c_void_p
    lib.kpool_score_topk_workspace_size_split.restype = ctypes.c_size_t
    lib.kpool_score_topk_workspace_size_split.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                          ctypes.c_int, ctypes.c_int]
    lib.kpool_score_topk_at.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_size_t, P]
    lib.kpool_last_error.restype = ctypes.c_char_p
    return lib


def _report(lib, call, res):
    out = (ctypes.c_ulonglong * 32)()
    call()
    torch.cuda.synchronize()
    lib.kpool_debug_phase_timers(out, 1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    call()
    e1.record()
    torch.cuda.synchronize()
    lib.kpool_debug_phase_timers(out, 1)
    v = list(out)
    res["ms"] = e0.elapsed_time(e1)
    for key, base, names in (("epilogue", 24, EPI), ("mma", 8, MMA), ("producer", 16, PROD)):
        tot = sum(v[base:base + 8]) or 1
        res[key] = {n: round(100.0 * v[base + i] / tot, 1) for i, n in enumerate(names)}
    return res


def run_decode(B_docs: int, lo: int, hi: int, H: int = 64, D: int = 128, kpool: int = 4,
               index_topk: int = 2048, seed: int = 0):
    lib = _lib()
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    lens = torch.randint(lo, hi, (B_docs,), generator=g, dtype=torch.int64)
    pools = lens // kpool
    cu_k = torch.zeros(B_docs + 1, dtype=torch.int32)
    cu_k[1:] = torch.cumsum(lens, 0).to(torch.int32)
    cu_p = torch.zeros(B_docs + 1, dtype=torch.int32)
    cu_p[1:] = torch.cumsum(pools, 0).to(torch.int32)
    P_total = int(cu_p[-1])
    cu_q = torch.arange(B_docs + 1, dtype=torch.int32)
    q_pos = (lens - 1).to(torch.int32)
    gd = torch.Generator(device="cuda")
    gd.manual_seed(seed)
    q = torch.randn(B_docs, H, D, device="cuda", generator=gd).to(torch.bfloat16)
    pk = torch.randn(P_total, D, device="cuda", generator=gd).to(torch.bfloat16)
    w = torch.randn(B_docs, H, device="cuda", generator=gd) / H ** 0.5
    Kp = index_topk // kpool
    idx = torch.empty(B_docs, Kp, dtype=torch.int32, device="cuda")
    sc = torch.empty(B_docs, Kp, dtype=torch.float32, device="cuda")
    nws = lib.kpool_score_topk_workspace_size_split(B_docs, H, B_docs, kpool, index_topk)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    d_cq, d_qp, d_cp = cu_q.cuda(), q_pos.cuda(), cu_p.cuda()
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())   # noqa: E731

    def call():
        rc = lib.kpool_score_topk_at(ptr(q), None, ptr(w), ptr(pk), None, ptr(d_cq), ptr(d_qp),
                                     ptr(d_cp), B_docs, B_docs, P_total, H, D, kpool, index_topk,
                                     0, ptr(idx), ptr(sc), ptr(ws), nws, None)
        if rc != 0:
            raise RuntimeError(lib.kpool_last_error())

    res = {"decode_docs": B_docs, "key_len": [lo, hi], "pools": P_total, "H": H, "D": D,
           "kpool": kpool, "index_topk": index_topk}
    return _report(lib, call, res)


def run(T: int, H: int = 64, D: int = 128, kpool: int = 4, index_topk: int = 2048, seed: int = 0,
        fp8: bool = False):
    lib = ctypes.CDLL(B.build(variant="phase_timers"))
    P = ctypes.c_void_p
    lib.kpool_score_topk_workspace_size.restype = ctypes.c_size_t
    lib.kpool_score_topk_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    lib.kpool_score_topk.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_size_t, P]
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q = torch.randn(T, H, D, device="cuda", generator=g).to(torch.bfloat16)
    pk = torch.randn(T // kpool, D, device="cuda", generator=g).to(torch.bfloat16)
    w = torch.randn(T, H, device="cuda", generator=g) / H ** 0.5
    qs = pks = None
    if fp8:
        lib.kpool_quantize_fp8.argtypes = [P, ctypes.c_int64, ctypes.c_int, P, P, P]
        q8 = torch.empty(T, H, D, dtype=torch.uint8, device="cuda")
        qs = torch.empty(T, H, dtype=torch.float32, device="cuda")
        pk8 = torch.empty(T // kpool, D, dtype=torch.uint8, device="cuda")
        pks = torch.empty(T // kpool, dtype=torch.float32, device="cuda")
        for src, dst, sc, rows in ((q, q8, qs, T * H), (pk, pk8, pks, T // kpool)):
            if lib.kpool_quantize_fp8(ctypes.c_void_p(src.data_ptr()), rows, D,
                                      ctypes.c_void_p(dst.data_ptr()),
                                      ctypes.c_void_p(sc.data_ptr()), None) != 0:
                raise RuntimeError("kpool_quantize_fp8 failed")
        q, pk = q8, pk8
    Kp = index_topk // kpool
    idx = torch.empty(T, Kp, dtype=torch.int32, device="cuda")
    sc = torch.empty(T, Kp, dtype=torch.float32, device="cuda")
    nws = lib.kpool_score_topk_workspace_size(T, H, 1)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())

    def call():
        rc = lib.kpool_score_topk(ptr(q), ptr(qs) if fp8 else None, ptr(w), ptr(pk),
                                  ptr(pks) if fp8 else None, None, None, 1, T, T // kpool, H, D,
                                  kpool, index_topk, int(fp8), ptr(idx), ptr(sc), ptr(ws), nws,
                                  None)
        if rc != 0:
            raise RuntimeError(lib.kpool_last_error())

    out = (ctypes.c_ulonglong * 32)()
    call()
    torch.cuda.synchronize()
    lib.kpool_debug_phase_timers(out, 1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    call()
    e1.record()
    torch.cuda.synchronize()
    lib.kpool_debug_phase_timers(out, 1)
    v = list(out)
    res = {"T": T, "H": H, "D": D, "kpool": kpool, "index_topk": index_topk, "fp8": fp8,
           "ms": e0.elapsed_time(e1)}
    for key, base, names in (("epilogue", 24, EPI), ("mma", 8, MMA), ("producer", 16, PROD)):
        tot = sum(v[base:base + 8]) or 1
        res[key] = {n: round(100.0 * v[base + i] / tot, 1) for i, n in enumerate(names)}
    return res


if __name__ == "__main__":
    for arg in sys.argv[1:] or ["131072"]:
        if arg.startswith("fp8:"):
            print(json.dumps(run(int(arg.split(":")[1]), fp8=True)))
        elif arg.startswith("decode:"):
            _, b, lo, hi = arg.split(":")
            print(json.dumps(run_decode(int(b), int(lo), int(hi))))
        else:
            print(json.dumps(run(int(arg))))
