"""kpool_indexer_forward_host (host buffers in, host token indices out, copies
overlapped with the kernels over query chunks) against the device path
kpool_indexer_forward on the same inputs: identical token indices, bit for
bit, for chunk sizes that cut through query tiles and documents; and against
the CPU oracle on sampled rows (selected pool sets equal up to near-tie
swaps, token rows bit-exact given the pools)."""
import numpy as np
import pytest
import torch

from sparse_attention_kpool_compress_gb300 import workloads as W
from kpool_checks import check_selection, pools_from_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_kpool_compress_gb300 as K
    return K


def _device_tokens(K, inp, wl, fp8):
    dev = torch.device("cuda")
    cu = inp.cu_seqlens
    multi = cu.numel() > 2
    cu_d = cp_d = P = None
    if multi:
        cp_h, P = K.kpool_num_pools(cu, wl.T, wl.kpool)
        cu_d, cp_d = cu.to(dev), cp_h.to(dev)
    tok, _, _ = K.kpool_indexer_forward(inp.q.to(dev), inp.k.to(dev), inp.gate.to(dev),
                                        inp.ape.to(dev), inp.w.to(dev), wl.kpool, wl.index_topk,
                                        wl.tail, cu_d, cp_d, P, fp8=fp8)
    torch.cuda.synchronize()
    return tok.cpu()


def _host_tokens(K, inp, wl, fp8, chunk_rows):
    pin = lambda x: x.contiguous().pin_memory()   # noqa: E731
    cu = inp.cu_seqlens if inp.cu_seqlens.numel() > 2 else None
    scratch = torch.empty(K.kpool_indexer_forward_host_scratch_size(
        wl.T, wl.H, wl.D, wl.kpool, wl.index_topk, cu, fp8, chunk_rows), dtype=torch.uint8,
        device="cuda")
    out = K.kpool_indexer_forward_host(pin(inp.q), pin(inp.k), pin(inp.gate), pin(inp.ape),
                                       pin(inp.w), wl.kpool, wl.index_topk, wl.tail, cu, fp8,
                                       chunk_rows, scratch=scratch)
    torch.cuda.synchronize()
    assert K.kpool_read_status(scratch) == 0
    return out


@pytest.mark.parametrize("chunk_rows", [3000, 4093, 0])
def test_single_sequence(K, chunk_rows):
    wl = W.Workload("p1", T=20000, H=64, D=128, kpool=4, index_topk=512)
    inp = W.make_inputs(wl, seed=31)
    assert torch.equal(_host_tokens(K, inp, wl, False, chunk_rows), _device_tokens(K, inp, wl, False))


def test_packed_documents_cut_by_chunks(K):
    wl = W.Workload("p2", T=12000, H=32, D=64, kpool=4, index_topk=256, n_docs=7,
                    doc_len_range=(100, 4000))
    inp = W.make_inputs(wl, seed=32)
    assert torch.equal(_host_tokens(K, inp, wl, False, 1000), _device_tokens(K, inp, wl, False))


def test_fp8_mode(K):
    wl = W.Workload("p3", T=9000, H=64, D=128, kpool=4, index_topk=1024, fp8=True)
    inp = W.make_inputs(wl, seed=33)
    assert torch.equal(_host_tokens(K, inp, wl, True, 2500), _device_tokens(K, inp, wl, True))


def test_no_tail_and_kpool_two(K):
    wl = W.Workload("p4", T=5000, H=16, D=128, kpool=2, index_topk=256, tail=False, n_docs=3,
                    doc_len_range=(500, 3000))
    inp = W.make_inputs(wl, seed=34)
    assert torch.equal(_host_tokens(K, inp, wl, False, 777), _device_tokens(K, inp, wl, False))


def test_no_complete_pool(K):
    wl = W.Workload("p5", T=3, H=4, D=32, kpool=4, index_topk=32)
    inp = W.make_inputs(wl, seed=35)
    out = _host_tokens(K, inp, wl, False, 0)
    assert torch.equal(out, _device_tokens(K, inp, wl, False))
    assert out[2, :3].tolist() == [0, 1, 2] and bool((out[:, 3:] == -1).all())


def test_packed_documents_fp8(K):
    """Packed documents and FP8 mode together: the per-chunk q quantisation and
    the per-document pooled-key scales across chunk boundaries."""
    wl = W.Workload("p6", T=10000, H=64, D=128, kpool=4, index_topk=512, n_docs=5,
                    doc_len_range=(500, 4000), fp8=True)
    inp = W.make_inputs(wl, seed=36)
    assert torch.equal(_host_tokens(K, inp, wl, True, 1500), _device_tokens(K, inp, wl, True))


def test_two_queries_per_warp_packed(K):
    """H = 32 (two queries per epilogue warp), packed documents, chunks of 999."""
    wl = W.Workload("p7", T=9000, H=32, D=128, kpool=4, index_topk=1024, n_docs=4,
                    doc_len_range=(800, 4000))
    inp = W.make_inputs(wl, seed=37)
    assert torch.equal(_host_tokens(K, inp, wl, False, 999), _device_tokens(K, inp, wl, False))


@pytest.mark.parametrize("packed", [False, True])
def test_host_pass_matches_oracle(K, ora, packed):
    """The host-buffer pass's token rows against the oracle on 256 sampled rows
    (plus the first and last 16): the pools the rows hold are the oracle's
    selection up to near-tie swaps (1e-3 * S of the Kp-th score), and each row
    is the oracle's expansion of those pools plus the causal tail."""
    if packed:
        wl = W.Workload("o2", T=12000, H=64, D=128, kpool=4, index_topk=512, n_docs=6,
                        doc_len_range=(300, 4000))
    else:
        wl = W.Workload("o1", T=16384, H=64, D=128, kpool=4, index_topk=512)
    inp = W.make_inputs(wl, seed=41 + int(packed))
    tok = _host_tokens(K, inp, wl, False, 3000).numpy()
    cu = inp.cu_seqlens.numpy() if packed else None
    rows = W.sample_rows(wl.T, n_sample=256, edge=16).numpy()
    pkb = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(), cu, wl.kpool)
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pkb)
    o = ora.select_rows(ops, cu, wl.kpool, wl.Kp, rows)
    pools = pools_from_tokens(tok[rows], rows, cu, wl.T, wl.kpool, o["n_sel"])
    idx = np.full((len(rows), wl.Kp), -1, np.int32)
    idx[:, : pools.shape[1]] = pools
    st = check_selection(ora, ops, cu, wl.kpool, wl.Kp, rows, idx, None, 1e-3, wl.name)
    assert st["swaps"] <= 4, st
    want = ora.expand_rows(idx, cu, wl.T, wl.kpool, wl.Kp, wl.tail, rows)
    assert np.array_equal(tok[rows], want)
