"""Python binding of libkpool.so (the GB300-native KPool DSA indexer).

Thin ctypes marshalling over the C ABI declared in ``include/kpool.h``: each
function checks dtypes/devices, allocates outputs with torch (device memory
and streams are torch's job here), and calls the C entry point of the same
name on the current CUDA stream.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback of any kind -- importing this
module fails loudly if ``libkpool.so`` has not been built.

Sources (page titles and sections): Megatron-LM PR "GLM5.3 Flash (KDA + mHC +
KPool DSA) support + FP8", Changes section 3 "KPool DSA indexer + NoPE";
SkyRL PR "GLM-5.3-Flash (glm5_next) Megatron support", commit "k-pool
indexer"; xtuner PR "GLM-5.3-Flash F5: NoPE DSA + KPool indexer".
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkpool.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libkpool.so is not built (expected at %s); run "
        "`python -c \"import __graft_entry__ as g; g.build()\"` or "
        "`python sparse_attention_kpool_compress_gb300/build.py`" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGS = {
    "kpool_last_error": (ctypes.c_char_p, []),
    "kpool_version": (_I, []),
    "kpool_num_pools": (_I, [_P, _I, _L, _I, _P, _P]),
    "kpool_cu_pools": (_I, [_P, _I, _I, _P, _P]),
    "kpool_compress": (_I, [_P, _P, _P, _P, _P, _I, _L, _I, _I, _L, _P, _P, _P, _P]),
    "kpool_quantize_fp8": (_I, [_P, _L, _I, _P, _P, _P]),
    "kpool_project_compress": (_I, [_P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _I, _L, _I, _I,
                                    _I, _L, _P, _P, _P, _P, _SZ, _P]),
    "kpool_score_topk_workspace_size": (_SZ, [_L, _I, _I]),
    "kpool_score_topk_workspace_size_split": (_SZ, [_L, _I, _I, _I, _I]),
    "kpool_score_topk": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _L, _L, _I, _I, _I, _I, _I,
                              _P, _P, _P, _SZ, _P]),
    "kpool_score_topk_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _L, _L, _I, _I, _I, _I,
                                      _I, _P, _P, _P]),
    "kpool_score_dense": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _L, _L, _I, _I, _I, _I,
                               _P, _P, _SZ, _P]),
    "kpool_expand_indices": (_I, [_P, _P, _P, _I, _L, _I, _I, _I, _P, _P]),
    "kpool_score_topk_at": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _L, _L, _I, _I, _I, _I, _I,
                                 _P, _P, _P, _SZ, _P]),
    "kpool_expand_indices_at": (_I, [_P, _P, _P, _P, _P, _I, _L, _I, _I, _I, _P, _P]),
    "kpool_sparse_mla_workspace_size": (_SZ, []),
    "kpool_sparse_mla_fwd": (_I, [_P, _P, _P, _L, _L, _I, _I, _I, ctypes.c_float, _P, _P, _P,
                                  _SZ, _P]),
    "kpool_sparse_mla_fwd_pools": (_I, [_P, _P, _P, _P, _P, _I, _L, _I, _I, _I, _I, _I,
                                        ctypes.c_float, _P, _P, _P, _SZ, _P]),
    "kpool_sparse_mla_fwd_pools_at": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _L, _L, _I, _I, _I,
                                           _I, _I, ctypes.c_float, _P, _P, _P, _SZ, _P]),
    "kpool_read_status": (_I, [_P, _P]),
    "kpool_score_topk_noalloc_status": (_I, [_P]),
    "kpool_debug_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "kpool_indexer_forward_host_scratch_size": (_SZ, [_P, _I, _L, _I, _I, _I, _I, _I, _L]),
    "kpool_indexer_forward_host": (_I, [_P, _P, _P, _P, _P, _P, _I, _L, _I, _I, _I, _I, _I, _I,
                                        _L, _P, _P, _SZ, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

STATUS_TIMEOUT = 1
STATUS_BAD_SEQLENS = 2


class KPoolError(RuntimeError):
    def __init__(self, code, fn):
        msg = _lib.kpool_last_error().decode(errors="replace")
        super().__init__("%s failed (%d): %s" % (fn, code, msg))
        self.code = code


def _check(rc, fn):
    if rc != 0:
        raise KPoolError(rc, fn)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype=None, device=True):
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    if device and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)


def _as_u8(t):
    if t is None:
        return None
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


def _docs(cu_seqlens, cu_pools):
    if cu_seqlens is None:
        if cu_pools is not None:
            raise ValueError("cu_pools given without cu_seqlens")
        return 1
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    _need(cu_pools, "cu_pools", torch.int32)
    return cu_seqlens.numel() - 1


# ---------------------------------------------------------------------------

def kpool_version() -> int:
    return int(_lib.kpool_version())


def kpool_num_pools(cu_seqlens_host, T: int, kpool: int):
    """Host helper: (cu_pools int32 CPU tensor, total pools) from a host
    cu_seqlens (list or CPU int32 tensor).  Validates the layout."""
    cs = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous().cpu()
    out = torch.empty_like(cs)
    total = ctypes.c_int64(0)
    _check(_lib.kpool_num_pools(_ptr(cs), cs.numel() - 1, T, kpool, _ptr(out),
                                ctypes.byref(total)), "kpool_num_pools")
    return out, int(total.value)


def kpool_cu_pools(cu_seqlens: torch.Tensor, kpool: int) -> torch.Tensor:
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    out = torch.empty_like(cu_seqlens)
    _check(_lib.kpool_cu_pools(_ptr(cu_seqlens), cu_seqlens.numel() - 1, kpool, _ptr(out),
                               _stream(cu_seqlens.device)), "kpool_cu_pools")
    return out


def kpool_compress(k, gate, ape, kpool: int, cu_seqlens=None, cu_pools=None, P_total=None,
                   fp8: bool = False, out=None):
    """Pooled keys pk [P_total, D] bf16 (plus E4M3 codes and scales when
    fp8).  For packed documents pass device cu_seqlens/cu_pools and P_total."""
    _need(k, "k", torch.bfloat16)
    _need(gate, "gate", torch.bfloat16)
    _need(ape, "ape", torch.float32)
    n_docs = _docs(cu_seqlens, cu_pools)
    T, D = k.shape
    if P_total is None:
        if cu_seqlens is not None:
            raise ValueError("P_total is required with cu_seqlens")
        P_total = T // kpool
    pk = out if out is not None else torch.empty(P_total, D, dtype=torch.bfloat16,
                                                 device=k.device)
    pk8 = sc = None
    if fp8:
        pk8 = torch.empty(P_total, D, dtype=torch.uint8, device=k.device)
        sc = torch.empty(P_total, dtype=torch.float32, device=k.device)
    _check(_lib.kpool_compress(_ptr(k), _ptr(gate), _ptr(ape), _ptr(cu_seqlens), _ptr(cu_pools),
                               n_docs, T, D, kpool, P_total, _ptr(pk), _ptr(pk8), _ptr(sc),
                               _stream(k.device)), "kpool_compress")
    return (pk, pk8, sc) if fp8 else pk


def kpool_project_compress(x, w_kg, k_norm_weight, k_norm_bias, k_norm_eps: float, ape,
                           kpool: int, cu_seqlens=None, cu_pools=None, P_total=None,
                           want_k_gate: bool = False, workspace=None):
    """Pooled keys pk [P_total, 128] bf16 straight from hidden states x [T,
    hidden] (key projection, k_norm, gate projection and compression in one
    kernel); with want_k_gate also the projected keys and gate [T, 128]."""
    _need(x, "x", torch.bfloat16)
    _need(w_kg, "w_kg", torch.bfloat16)
    for t_, n_ in ((k_norm_weight, "k_norm_weight"), (k_norm_bias, "k_norm_bias"), (ape, "ape")):
        _need(t_, n_, torch.float32)
    n_docs = _docs(cu_seqlens, cu_pools)
    T, hidden = x.shape
    D = w_kg.shape[0] // 2
    if P_total is None:
        if cu_seqlens is not None:
            raise ValueError("P_total is required with cu_seqlens")
        P_total = T // kpool
    pk = torch.empty(P_total, D, dtype=torch.bfloat16, device=x.device)
    k_out = g_out = None
    if want_k_gate:
        k_out = torch.empty(T, D, dtype=torch.bfloat16, device=x.device)
        g_out = torch.empty(T, D, dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(256, dtype=torch.uint8, device=x.device)
    _check(_lib.kpool_project_compress(_ptr(x), _ptr(w_kg), _ptr(k_norm_weight),
                                       _ptr(k_norm_bias), float(k_norm_eps), _ptr(ape),
                                       _ptr(cu_seqlens), _ptr(cu_pools), n_docs, T, hidden, D,
                                       kpool, P_total, _ptr(pk), _ptr(k_out), _ptr(g_out),
                                       _ptr(workspace), workspace.numel(), _stream(x.device)),
           "kpool_project_compress")
    return (pk, k_out, g_out) if want_k_gate else pk


def kpool_quantize_fp8(x):
    """x bf16 [..., 128] -> (E4M3 codes uint8 [..., 128], fp32 scales [...])."""
    _need(x, "x", torch.bfloat16)
    D = x.shape[-1]
    rows = x.numel() // D
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    sc = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _check(_lib.kpool_quantize_fp8(_ptr(x), rows, D, _ptr(codes), _ptr(sc), _stream(x.device)),
           "kpool_quantize_fp8")
    return codes, sc


def kpool_score_topk_workspace_size(T: int, H: int, n_docs: int = 1) -> int:
    return int(_lib.kpool_score_topk_workspace_size(T, H, n_docs))


def kpool_score_topk_workspace_size_split(T: int, H: int, n_docs: int, kpool: int,
                                          index_topk: int) -> int:
    return int(_lib.kpool_score_topk_workspace_size_split(T, H, n_docs, kpool, index_topk))


def new_workspace(T: int, H: int, n_docs: int = 1, device="cuda", kpool: int | None = None,
                  index_topk: int | None = None) -> torch.Tensor:
    """Workspace for kpool_score_topk[_at]; with kpool and index_topk it is
    large enough for the split-pool schedule of calls with few query tiles."""
    if kpool is not None and index_topk is not None:
        n = kpool_score_topk_workspace_size_split(T, H, n_docs, kpool, index_topk)
    else:
        n = kpool_score_topk_workspace_size(T, H, n_docs)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def _score_common(q, w, pk, q_scale, pk_scale, cu_seqlens, cu_pools):
    fp8 = q_scale is not None
    if fp8:
        _need(q, "q", (torch.uint8, torch.float8_e4m3fn))
        _need(pk, "pk", (torch.uint8, torch.float8_e4m3fn))
        _need(q_scale, "q_scale", torch.float32)
        _need(pk_scale, "pk_scale", torch.float32)
    else:
        _need(q, "q", torch.bfloat16)
        _need(pk, "pk", torch.bfloat16)
    _need(w, "w", torch.float32)
    n_docs = _docs(cu_seqlens, cu_pools)
    T, H, D = q.shape
    return fp8, n_docs, T, H, D, pk.shape[0]


def kpool_score_topk(q, w, pk, kpool: int, index_topk: int, cu_seqlens=None, cu_pools=None,
                     q_scale=None, pk_scale=None, workspace=None, out=None):
    """(pool_idx int32 [T, Kp], pool_score fp32 [T, Kp]) -- ascending pools,
    -1 / -inf padded."""
    fp8, n_docs, T, H, D, P = _score_common(q, w, pk, q_scale, pk_scale, cu_seqlens, cu_pools)
    Kp = index_topk // kpool
    if workspace is None:
        workspace = new_workspace(T, H, n_docs, q.device, kpool, index_topk)
    if out is None:
        idx = torch.empty(T, Kp, dtype=torch.int32, device=q.device)
        sc = torch.empty(T, Kp, dtype=torch.float32, device=q.device)
    else:
        idx, sc = out
    _check(_lib.kpool_score_topk(_ptr(_as_u8(q)) if fp8 else _ptr(q), _ptr(q_scale), _ptr(w),
                                 _ptr(_as_u8(pk)) if fp8 else _ptr(pk), _ptr(pk_scale),
                                 _ptr(cu_seqlens), _ptr(cu_pools), n_docs, T, P, H, D, kpool,
                                 index_topk, int(fp8), _ptr(idx), _ptr(sc), _ptr(workspace),
                                 workspace.numel(), _stream(q.device)), "kpool_score_topk")
    return idx, sc


def kpool_score_topk_noalloc(q, w, pk, kpool: int, index_topk: int, cu_seqlens=None,
                             cu_pools=None, q_scale=None, pk_scale=None, out=None):
    """kpool_score_topk without a workspace: the library's fixed scratch
    array stands in for it (see include/kpool.h for its limits)."""
    fp8, n_docs, T, H, D, P = _score_common(q, w, pk, q_scale, pk_scale, cu_seqlens, cu_pools)
    Kp = index_topk // kpool
    if out is None:
        idx = torch.empty(T, Kp, dtype=torch.int32, device=q.device)
        sc = torch.empty(T, Kp, dtype=torch.float32, device=q.device)
    else:
        idx, sc = out
    _check(_lib.kpool_score_topk_noalloc(_ptr(_as_u8(q)) if fp8 else _ptr(q), _ptr(q_scale),
                                         _ptr(w), _ptr(_as_u8(pk)) if fp8 else _ptr(pk),
                                         _ptr(pk_scale), _ptr(cu_seqlens), _ptr(cu_pools), n_docs,
                                         T, P, H, D, kpool, index_topk, int(fp8), _ptr(idx),
                                         _ptr(sc), _stream(q.device)),
           "kpool_score_topk_noalloc")
    return idx, sc


def kpool_score_dense(q, w, pk, kpool: int, cu_seqlens=None, cu_pools=None, q_scale=None,
                      pk_scale=None, workspace=None):
    """Test/debug: full fp32 [T, P] scores (-inf where not a causal pool)."""
    fp8, n_docs, T, H, D, P = _score_common(q, w, pk, q_scale, pk_scale, cu_seqlens, cu_pools)
    if workspace is None:
        workspace = new_workspace(T, H, n_docs, q.device)
    out = torch.empty(T, P, dtype=torch.float32, device=q.device)
    _check(_lib.kpool_score_dense(_ptr(_as_u8(q)) if fp8 else _ptr(q), _ptr(q_scale), _ptr(w),
                                  _ptr(_as_u8(pk)) if fp8 else _ptr(pk), _ptr(pk_scale),
                                  _ptr(cu_seqlens), _ptr(cu_pools), n_docs, T, P, H, D, kpool,
                                  int(fp8), _ptr(out), _ptr(workspace), workspace.numel(),
                                  _stream(q.device)), "kpool_score_dense")
    return out


def kpool_expand_indices(pool_idx, kpool: int, index_topk: int, always_select_tail: bool = True,
                         cu_seqlens=None, cu_pools=None, out=None):
    """Token indices int32 [T, Kp*kpool + kpool - 1], ascending, -1 padded."""
    _need(pool_idx, "pool_idx", torch.int32)
    n_docs = _docs(cu_seqlens, cu_pools)
    T = pool_idx.shape[0]
    Kp = index_topk // kpool
    W = Kp * kpool + kpool - 1
    tok = out if out is not None else torch.empty(T, W, dtype=torch.int32, device=pool_idx.device)
    _check(_lib.kpool_expand_indices(_ptr(pool_idx), _ptr(cu_seqlens), _ptr(cu_pools), n_docs, T,
                                     kpool, index_topk, int(bool(always_select_tail)), _ptr(tok),
                                     _stream(pool_idx.device)), "kpool_expand_indices")
    return tok


def kpool_score_topk_at(q, w, pk, kpool: int, index_topk: int, cu_seqlens_q, q_start_pos,
                        cu_pools, q_scale=None, pk_scale=None, workspace=None, out=None):
    """Positioned queries (decode / chunked prefill): document d's query rows
    [cu_seqlens_q[d], cu_seqlens_q[d+1]) sit at positions q_start_pos[d] + i."""
    fp8, n_docs, T, H, D, P = _score_common(q, w, pk, q_scale, pk_scale, cu_seqlens_q, cu_pools)
    _need(q_start_pos, "q_start_pos", torch.int32)
    Kp = index_topk // kpool
    if workspace is None:
        workspace = new_workspace(T, H, n_docs, q.device, kpool, index_topk)
    if out is None:
        idx = torch.empty(T, Kp, dtype=torch.int32, device=q.device)
        sc = torch.empty(T, Kp, dtype=torch.float32, device=q.device)
    else:
        idx, sc = out
    _check(_lib.kpool_score_topk_at(_ptr(_as_u8(q)) if fp8 else _ptr(q), _ptr(q_scale), _ptr(w),
                                    _ptr(_as_u8(pk)) if fp8 else _ptr(pk), _ptr(pk_scale),
                                    _ptr(cu_seqlens_q), _ptr(q_start_pos), _ptr(cu_pools), n_docs,
                                    T, P, H, D, kpool, index_topk, int(fp8), _ptr(idx), _ptr(sc),
                                    _ptr(workspace), workspace.numel(), _stream(q.device)),
           "kpool_score_topk_at")
    return idx, sc


def kpool_expand_indices_at(pool_idx, kpool: int, index_topk: int, cu_seqlens_q, q_start_pos,
                            cu_seqlens_k, cu_pools, always_select_tail: bool = True, out=None):
    """Key-token indices for positioned queries [Tq, Kp*kpool + kpool - 1]."""
    _need(pool_idx, "pool_idx", torch.int32)
    for t_, n_ in ((cu_seqlens_q, "cu_seqlens_q"), (q_start_pos, "q_start_pos"),
                   (cu_seqlens_k, "cu_seqlens_k"), (cu_pools, "cu_pools")):
        _need(t_, n_, torch.int32)
    T = pool_idx.shape[0]
    Kp = index_topk // kpool
    W = Kp * kpool + kpool - 1
    tok = out if out is not None else torch.empty(T, W, dtype=torch.int32, device=pool_idx.device)
    _check(_lib.kpool_expand_indices_at(_ptr(pool_idx), _ptr(cu_seqlens_q), _ptr(q_start_pos),
                                        _ptr(cu_seqlens_k), _ptr(cu_pools), cu_seqlens_q.numel() - 1,
                                        T, kpool, index_topk, int(bool(always_select_tail)),
                                        _ptr(tok), _stream(pool_idx.device)),
           "kpool_expand_indices_at")
    return tok


def kpool_sparse_mla_workspace_size() -> int:
    return int(_lib.kpool_sparse_mla_workspace_size())


def _mla_outputs(q, workspace, o, lse):
    T, H, Dc = q.shape
    if o is None:
        o = torch.empty(T, H, Dc, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(T, H, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(kpool_sparse_mla_workspace_size(), dtype=torch.uint8,
                                device=q.device)
    return o, lse, workspace


def kpool_sparse_mla_fwd(q, kv, tok_idx, softmax_scale: float, workspace=None, o=None, lse=None):
    """Sparse attention over explicit token lists: q bf16 [T, 64, 512], kv bf16
    [Tk, 512], tok_idx int32 [T, W] (-1 = none) -> (o bf16 [T, 64, 512], lse
    fp32 [T, 64])."""
    _need(q, "q", torch.bfloat16)
    _need(kv, "kv", torch.bfloat16)
    _need(tok_idx, "tok_idx", torch.int32)
    T, H, Dc = q.shape
    o, lse, workspace = _mla_outputs(q, workspace, o, lse)
    _check(_lib.kpool_sparse_mla_fwd(_ptr(q), _ptr(kv), _ptr(tok_idx), T, kv.shape[0],
                                     tok_idx.shape[1], H, Dc, float(softmax_scale), _ptr(o),
                                     _ptr(lse), _ptr(workspace), workspace.numel(),
                                     _stream(q.device)), "kpool_sparse_mla_fwd")
    return o, lse


def kpool_sparse_mla_fwd_pools(q, kv, pool_idx, kpool: int, index_topk: int,
                               softmax_scale: float, cu_seqlens=None, cu_pools=None,
                               always_select_tail: bool = True, workspace=None, o=None, lse=None):
    """Sparse attention fused with the expansion of pool_idx [T, index_topk //
    kpool] (keys = the query tokens, kv bf16 [T, 512])."""
    _need(q, "q", torch.bfloat16)
    _need(kv, "kv", torch.bfloat16)
    _need(pool_idx, "pool_idx", torch.int32)
    n_docs = _docs(cu_seqlens, cu_pools)
    T, H, Dc = q.shape
    o, lse, workspace = _mla_outputs(q, workspace, o, lse)
    _check(_lib.kpool_sparse_mla_fwd_pools(_ptr(q), _ptr(kv), _ptr(pool_idx), _ptr(cu_seqlens),
                                           _ptr(cu_pools), n_docs, T, H, Dc, kpool, index_topk,
                                           int(bool(always_select_tail)), float(softmax_scale),
                                           _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(),
                                           _stream(q.device)), "kpool_sparse_mla_fwd_pools")
    return o, lse


def kpool_sparse_mla_fwd_pools_at(q, kv, pool_idx, kpool: int, index_topk: int,
                                  softmax_scale: float, cu_seqlens_q, q_start_pos, cu_seqlens_k,
                                  cu_pools, always_select_tail: bool = True, workspace=None,
                                  o=None, lse=None):
    """kpool_sparse_mla_fwd_pools for positioned queries (keys kv [Tk, 512])."""
    _need(q, "q", torch.bfloat16)
    _need(kv, "kv", torch.bfloat16)
    _need(pool_idx, "pool_idx", torch.int32)
    for t_, n_ in ((cu_seqlens_q, "cu_seqlens_q"), (q_start_pos, "q_start_pos"),
                   (cu_seqlens_k, "cu_seqlens_k"), (cu_pools, "cu_pools")):
        _need(t_, n_, torch.int32)
    T, H, Dc = q.shape
    o, lse, workspace = _mla_outputs(q, workspace, o, lse)
    _check(_lib.kpool_sparse_mla_fwd_pools_at(
        _ptr(q), _ptr(kv), _ptr(pool_idx), _ptr(cu_seqlens_q), _ptr(q_start_pos),
        _ptr(cu_seqlens_k), _ptr(cu_pools), cu_seqlens_q.numel() - 1, T, kv.shape[0], H, Dc,
        kpool, index_topk, int(bool(always_select_tail)), float(softmax_scale), _ptr(o),
        _ptr(lse), _ptr(workspace), workspace.numel(), _stream(q.device)),
        "kpool_sparse_mla_fwd_pools_at")
    return o, lse


def _host_cu(cu_seqlens_host):
    if cu_seqlens_host is None:
        return None, 1
    _need(cu_seqlens_host, "cu_seqlens_host", torch.int32, device=False)
    if cu_seqlens_host.is_cuda:
        raise ValueError("cu_seqlens_host must be a CPU tensor")
    return cu_seqlens_host, cu_seqlens_host.numel() - 1


def kpool_indexer_forward_host_scratch_size(T: int, H: int, D: int, kpool: int, index_topk: int,
                                            cu_seqlens_host=None, fp8: bool = False,
                                            chunk_rows: int = 0) -> int:
    cu, n_docs = _host_cu(cu_seqlens_host)
    return int(_lib.kpool_indexer_forward_host_scratch_size(_ptr(cu), n_docs, T, H, D, kpool,
                                                            index_topk, int(fp8), chunk_rows))


def kpool_indexer_forward_host(q, k, gate, ape, w, kpool: int, index_topk: int,
                               always_select_tail: bool = True, cu_seqlens_host=None,
                               fp8: bool = False, chunk_rows: int = 0, scratch=None, out=None,
                               device=None):
    """The whole pass from host (CPU, ideally pinned) tensors to host token
    indices int32 [T, Kp*kpool + kpool - 1], copies overlapped with the
    kernels.  Enqueued on the current CUDA stream of `device`; synchronize it
    before reading the result.  Without `scratch`, a device scratch of
    kpool_indexer_forward_host_scratch_size bytes (about 0.9 GB at T=131072)
    is allocated for the call: pass one to reuse it across calls."""
    for t_, n_, dt in ((q, "q", torch.bfloat16), (k, "k", torch.bfloat16),
                       (gate, "gate", torch.bfloat16), (ape, "ape", torch.float32),
                       (w, "w", torch.float32)):
        _need(t_, n_, dt, device=False)
        if t_.is_cuda:
            raise ValueError("%s must be a host tensor" % n_)
    cu, n_docs = _host_cu(cu_seqlens_host)
    T, H, D = q.shape
    dev = torch.device("cuda") if device is None else torch.device(device)
    W = (index_topk // kpool) * kpool + kpool - 1
    if out is None:
        out = torch.empty(T, W, dtype=torch.int32, pin_memory=True)
    if scratch is None:
        n = kpool_indexer_forward_host_scratch_size(T, H, D, kpool, index_topk, cu, fp8,
                                                    chunk_rows)
        scratch = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    _check(_lib.kpool_indexer_forward_host(_ptr(q), _ptr(k), _ptr(gate), _ptr(ape), _ptr(w),
                                           _ptr(cu), n_docs, T, H, D, kpool, index_topk,
                                           int(bool(always_select_tail)), int(fp8), chunk_rows,
                                           _ptr(out), _ptr(scratch), scratch.numel(),
                                           _stream(dev)), "kpool_indexer_forward_host")
    return out


def kpool_read_status(workspace) -> int:
    v = ctypes.c_int(0)
    _check(_lib.kpool_read_status(_ptr(workspace), ctypes.byref(v)), "kpool_read_status")
    return int(v.value)


def kpool_score_topk_noalloc_status() -> int:
    """Status word of the last kpool_score_topk_noalloc on the current device."""
    v = ctypes.c_int(0)
    _check(_lib.kpool_score_topk_noalloc_status(ctypes.byref(v)),
           "kpool_score_topk_noalloc_status")
    return int(v.value)


def kpool_debug_set_wait_limit_ns(ns: int) -> int:
    """Test entry: limit of each scoring-kernel wait (0 = the 2 s default);
    returns the previous limit."""
    return int(_lib.kpool_debug_set_wait_limit_ns(int(ns)))


def kpool_indexer_forward(q, k, gate, ape, w, kpool: int, index_topk: int,
                          always_select_tail: bool = True, cu_seqlens=None, cu_pools=None,
                          P_total=None, fp8: bool = False, workspace=None):
    """The whole indexer path on the current stream: compress -> (FP8 cast of
    q and pooled keys) -> score + top-k -> expand.  Returns
    (tok_idx, pool_idx, pool_score)."""
    if fp8:
        pk, pk8, pks = kpool_compress(k, gate, ape, kpool, cu_seqlens, cu_pools, P_total, fp8=True)
        q8, qs = kpool_quantize_fp8(q)
        idx, sc = kpool_score_topk(q8, w, pk8, kpool, index_topk, cu_seqlens, cu_pools,
                                   q_scale=qs, pk_scale=pks, workspace=workspace)
    else:
        pk = kpool_compress(k, gate, ape, kpool, cu_seqlens, cu_pools, P_total)
        idx, sc = kpool_score_topk(q, w, pk, kpool, index_topk, cu_seqlens, cu_pools,
                                   workspace=workspace)
    tok = kpool_expand_indices(idx, kpool, index_topk, always_select_tail, cu_seqlens, cu_pools)
    return tok, idx, sc


__all__ = [n for n in dir() if n.startswith("kpool_")] + ["KPoolError", "new_workspace",
                                                           "LIB_PATH"]
