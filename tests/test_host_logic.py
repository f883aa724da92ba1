"""Host-side logic without a GPU: query layouts of the positioned workloads
and the benchmark's per-row pool counts."""
import numpy as np

from sparse_attention_kpool_compress_gb300 import workloads as W


def test_query_layout_prefill_is_none():
    assert W.query_layout("all", [5, 7]) is None


def test_query_layout_decode_last_key():
    cu_q, q_pos = W.query_layout("last", [5, 7, 1])
    assert cu_q == [0, 1, 2, 3]
    assert q_pos == [4, 6, 0]


def test_query_layout_chunk_clipped_to_document():
    cu_q, q_pos = W.query_layout("chunk:4", [10, 3, 4])
    assert cu_q == [0, 4, 7, 11]
    assert q_pos == [6, 0, 0]


def test_positioned_inputs_shapes():
    wl = W.Workload("p", T=96, H=2, D=32, kpool=4, index_topk=8, n_docs=3,
                    doc_len_range=(16, 48), queries="chunk:5")
    inp = W.make_inputs(wl)
    lens = np.diff(inp.cu_seqlens.numpy())
    assert inp.Tq == int(np.minimum(lens, 5).sum())
    assert inp.q.shape == (inp.Tq, 2, 32) and inp.w.shape == (inp.Tq, 2)
    assert inp.k.shape == (96, 32)
    assert np.array_equal(inp.q_pos.numpy(), lens - np.minimum(lens, 5))


def test_positioned_counts_match_brute_force():
    import bench
    wl = W.Workload("p", T=200, H=2, D=32, kpool=4, index_topk=8, n_docs=4,
                    doc_len_range=(10, 90), queries="chunk:7")
    inp = W.make_inputs(wl)
    nc = bench.positioned_counts(inp)
    cu_k, cq, qp = inp.cu_seqlens.numpy(), inp.cu_q.numpy(), inp.q_pos.numpy()
    want = []
    for d in range(4):
        L = cu_k[d + 1] - cu_k[d]
        for i in range(cq[d + 1] - cq[d]):
            tau = qp[d] + i
            # complete pools whose last token is at or before tau
            want.append(sum(1 for j in range(L // 4) if 4 * j + 3 <= tau))
    assert nc.tolist() == want


def test_chunk_compress_plan():
    import bench
    inp = W.make_inputs(W.Workload("c", T=64, H=2, D=32, kpool=4, index_topk=8,
                                   queries="chunk:16"))
    assert bench.chunk_compress_plan(inp) == (48, 12)
    inp = W.make_inputs(W.Workload("c", T=64, H=2, D=32, kpool=4, index_topk=8,
                                   queries="chunk:15"))
    assert bench.chunk_compress_plan(inp) is None      # not on a pool boundary
    inp = W.make_inputs(W.Workload("d", T=64, H=2, D=32, kpool=4, index_topk=8, n_docs=2,
                                   equal_docs=True, queries="last"))
    assert bench.chunk_compress_plan(inp) is None


def test_source_fingerprint_ignores_comments(tmp_path):
    import bench
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("int f(int x) {\n  return x + 1;  // one\n}\n")
    b.write_text("/* header */\nint f(int x)\n{\n    return x + 1;\n}\n")
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.file_hash(str(a)) == bench.file_hash(str(b))
    assert bench.file_hash(str(a)) != bench.file_hash(str(c))


def test_reference_arm_positioned_workload(capsys, monkeypatch):
    """The oracle arm on a tiny decode-style workload: one JSON line with the
    reference fields (the oracle times selection and expansion of the rows)."""
    import json
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)

    class A:
        steps = 1
        warmup = 3
        ref_rows = 8
    wl = W.Workload("tiny_decode", T=600, H=4, D=32, kpool=4, index_topk=32, n_docs=3,
                    doc_len_range=(100, 300), queries="last")
    assert bench.run_reference(A(), wl) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert "pooled-key cache" in line["cpu_baseline"]["sample"]
