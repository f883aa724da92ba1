"""C-ABI checks that need no GPU: the library builds/loads, exports every
symbol include/kpool.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kpool.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_kpool_compress_gb300 import build as B
    path = B.build()
    return ctypes.CDLL(path)


def declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"KPOOL_API\s+[\w\s\*]+?\b(kpool_\w+)\s*\(", src)))


def test_header_declares_entry_points():
    syms = declared_symbols()
    for need in ["kpool_compress", "kpool_score_topk", "kpool_expand_indices",
                 "kpool_quantize_fp8", "kpool_num_pools", "kpool_score_dense",
                 "kpool_score_topk_workspace_size", "kpool_last_error", "kpool_read_status",
                 "kpool_cu_pools", "kpool_version"]:
        assert need in syms


def test_library_exports_every_declared_symbol(lib):
    from sparse_attention_kpool_compress_gb300 import build as B
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (kpool_\w+)", out))
    for s in declared_symbols():
        assert s in exported, s
        assert hasattr(lib, s)


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "kpool.h"\nint main(void){return kpool_version() > 0 ? 0 : 1;}\n')
    r = subprocess.run(["gcc", "-std=c99", "-fsyntax-only", "-I", os.path.dirname(HEADER),
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_binding_names_match_abi():
    import sparse_attention_kpool_compress_gb300 as K
    from sparse_attention_kpool_compress_gb300 import binding
    for s in declared_symbols():
        if s in ("kpool_last_error",):
            continue
        assert hasattr(binding, s), s


def test_version_and_workspace(lib):
    import sparse_attention_kpool_compress_gb300 as K
    assert K.kpool_version() == 10000
    assert K.kpool_score_topk_workspace_size(131072, 64, 1) >= 8 * 131072 // 4
    assert K.kpool_score_topk_workspace_size(0, 64, 1) > 0
    assert K.kpool_score_topk_workspace_size(100, 7, 1) == 0     # unsupported H


def test_num_pools_host_helper():
    import sparse_attention_kpool_compress_gb300 as K
    cp, total = K.kpool_num_pools([0, 10, 27, 27, 64], 64, 4)
    assert cp.tolist() == [0, 2, 6, 6, 15] and total == 15
    for bad in ([1, 10, 64], [0, 10, 5, 64], [0, 10, 63]):
        with pytest.raises(K.KPoolError) as e:
            K.kpool_num_pools(bad, 64, 4)
        assert e.value.code == -1
    with pytest.raises(K.KPoolError):
        K.kpool_num_pools([0, 64], 64, 0)


P = ctypes.c_void_p


def _fake(n=1 << 20):
    """A host buffer whose address stands in for a device pointer: only ever
    passed to calls that must reject their arguments before any launch."""
    buf = ctypes.create_string_buffer(n + 512)
    addr = (ctypes.addressof(buf) + 255) & ~255
    return buf, ctypes.c_void_p(addr)


def test_host_validation_rejects_bad_arguments(lib):
    from sparse_attention_kpool_compress_gb300 import binding as b
    L = b._lib
    keep, p = _fake()
    _, p_mis = None, ctypes.c_void_p(p.value + 2)
    ws_n = L.kpool_score_topk_workspace_size(1024, 64, 1)
    cases = [
        # kpool_compress: D unsupported, kpool 0, misaligned k, P_total mismatch
        (L.kpool_compress, (p, p, p, None, None, 1, 1024, 96, 4, 256, p, None, None, None), -2),
        (L.kpool_compress, (p, p, p, None, None, 1, 1024, 128, 0, 256, p, None, None, None), -2),
        (L.kpool_compress, (p_mis, p, p, None, None, 1, 1024, 128, 4, 256, p, None, None, None), -1),
        (L.kpool_compress, (p, p, p, None, None, 1, 1024, 128, 4, 100, p, None, None, None), -1),
        (L.kpool_compress, (p, p, p, p, None, 1, 1024, 128, 4, 256, p, None, None, None), -1),
        (L.kpool_compress, (p, p, p, None, None, 1, 1024, 64, 4, 256, p, p, p, None), -2),
        # kpool_quantize_fp8: D != 128
        (L.kpool_quantize_fp8, (p, 16, 64, p, p, None), -2),
        # kpool_score_topk: H unsupported, index_topk % kpool, workspace too small,
        # Kp above capacity, fp8 without scales, D unsupported
        (L.kpool_score_topk, (p, None, p, p, None, None, None, 1, 1024, 256, 48, 128, 4, 2048, 0,
                              p, p, p, ws_n, None), -2),
        (L.kpool_score_topk, (p, None, p, p, None, None, None, 1, 1024, 256, 64, 128, 4, 2047, 0,
                              p, p, p, ws_n, None), -1),
        (L.kpool_score_topk, (p, None, p, p, None, None, None, 1, 1024, 256, 64, 128, 4, 2048, 0,
                              p, p, p, 16, None), -4),
        (L.kpool_score_topk, (p, None, p, p, None, None, None, 1, 1024, 256, 64, 128, 4, 1 << 16,
                              0, p, p, p, ws_n, None), -2),
        (L.kpool_score_topk, (p, None, p, p, None, None, None, 1, 1024, 256, 64, 128, 4, 2048, 1,
                              p, p, p, ws_n, None), -1),
        (L.kpool_score_topk, (p, None, p, p, None, None, None, 1, 1024, 256, 64, 96, 4, 2048, 0,
                              p, p, p, ws_n, None), -2),
        (L.kpool_score_topk, (p_mis, None, p, p, None, None, None, 1, 1024, 256, 64, 128, 4, 2048,
                              0, p, p, p, ws_n, None), -1),
        # kpool_expand_indices: index_topk not a multiple of kpool; n_docs without cu_seqlens
        (L.kpool_expand_indices, (p, None, None, 1, 1024, 4, 2046, 1, p, None), -1),
        (L.kpool_expand_indices, (p, None, None, 2, 1024, 4, 2048, 1, p, None), -1),
        # kpool_sparse_mla_fwd: heads / latent width outside the built shape, scale <= 0,
        # misaligned q, short workspace, negative width, no token list
        (L.kpool_sparse_mla_fwd, (p, p, p, 16, 16, 4, 32, 512, 0.1, p, p, p, 256, None), -2),
        (L.kpool_sparse_mla_fwd, (p, p, p, 16, 16, 4, 64, 256, 0.1, p, p, p, 256, None), -2),
        (L.kpool_sparse_mla_fwd, (p, p, p, 16, 16, 4, 64, 512, 0.0, p, p, p, 256, None), -1),
        (L.kpool_sparse_mla_fwd, (p_mis, p, p, 16, 16, 4, 64, 512, 0.1, p, p, p, 256, None), -1),
        (L.kpool_sparse_mla_fwd, (p, p, p, 16, 16, 4, 64, 512, 0.1, p, p, p, 16, None), -4),
        (L.kpool_sparse_mla_fwd, (p, p, p, 16, 16, -1, 64, 512, 0.1, p, p, p, 256, None), -1),
        (L.kpool_sparse_mla_fwd, (p, p, None, 16, 16, 4, 64, 512, 0.1, p, p, p, 256, None), -1),
        # kpool_sparse_mla_fwd_pools: index_topk not a multiple of kpool, n_docs without
        # cu_seqlens; _pools_at: missing per-document arrays
        (L.kpool_sparse_mla_fwd_pools, (p, p, p, None, None, 1, 16, 64, 512, 4, 2046, 1, 0.1,
                                        p, p, p, 256, None), -1),
        (L.kpool_sparse_mla_fwd_pools, (p, p, p, None, None, 2, 16, 64, 512, 4, 2048, 1, 0.1,
                                        p, p, p, 256, None), -1),
        (L.kpool_sparse_mla_fwd_pools_at, (p, p, p, None, p, p, p, 1, 16, 16, 64, 512, 4, 2048, 1,
                                           0.1, p, p, p, 256, None), -1),
    ]
    for fn, args, code in cases:
        rc = fn(*args)
        assert rc == code, (fn.__name__, rc, L.kpool_last_error())
        assert L.kpool_last_error()
    del keep


def test_host_pipeline_sizes_and_validation():
    """kpool_indexer_forward_host: scratch size 0 for unsupported shapes,
    layout errors caught on the host before any device work."""
    import ctypes
    import sparse_attention_kpool_compress_gb300 as K
    assert K.kpool_indexer_forward_host_scratch_size(4096, 64, 128, 4, 2048) > 0
    assert K.kpool_indexer_forward_host_scratch_size(4096, 7, 128, 4, 2048) == 0      # H
    assert K.kpool_indexer_forward_host_scratch_size(4096, 64, 96, 4, 2048) == 0      # D
    assert K.kpool_indexer_forward_host_scratch_size(4096, 64, 64, 4, 2048, fp8=True) == 0
    assert K.kpool_indexer_forward_host_scratch_size(4096, 64, 128, 4, 2047) == 0     # topk
    a = K.kpool_indexer_forward_host_scratch_size(4096, 64, 128, 4, 2048, chunk_rows=1024)
    b = K.kpool_indexer_forward_host_scratch_size(4096, 64, 128, 4, 2048, chunk_rows=2048)
    assert 0 < a < b
    L = K.binding._lib
    bad = (ctypes.c_int32 * 3)(0, 10, 5)          # decreasing offsets
    dummy = ctypes.c_void_p(16)
    rc = L.kpool_indexer_forward_host(dummy, dummy, dummy, dummy, dummy,
                                      ctypes.cast(bad, ctypes.c_void_p), 2, 5, 64, 128, 4, 2048,
                                      1, 0, 0, dummy, ctypes.c_void_p(256), 1 << 20, None)
    assert rc == -1                                # KPOOL_ERR_INVALID_ARG
    rc = L.kpool_indexer_forward_host(dummy, dummy, dummy, dummy, dummy, None, 1, 5, 64, 128, 4,
                                      2048, 1, 0, -1, dummy, ctypes.c_void_p(256), 1 << 20, None)
    assert rc == -1                                # negative chunk_rows
