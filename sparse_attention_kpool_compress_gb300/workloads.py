"""Seeded synthetic inputs for the KPool indexer.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so the CUDA path and the CPU oracle can both take their
inputs from it.  Draw order and distributions (seed 0 by default, a
``torch.Generator``):

1. document lengths (packed-THD workloads only): ``u_i ~ U[lo, hi)`` in
   float64, ``L_i = floor(u_i * T / sum(u))``, the remainder added to the
   last document;
2. ``q [Tq, H, D]``, 3. ``k [T, D]``, 4. ``gate [T, D]``: N(0, 1) drawn in
   float32 and rounded to bfloat16 by torch;
5. ``ape [kpool, D]``: N(0, 0.1^2) float32;
6. ``w [Tq, H]``: N(0, 1) / sqrt(H) float32.

``T`` counts key tokens.  A prefill (``queries="all"``) has one query per
key, ``Tq = T``.  Positioned workloads have fewer queries, the last ones of
each document: ``"last"`` is one decode query per document (at the document's
last key), ``"chunk:N"`` the final chunk of N tokens of a chunked prefill.
Their query rows are described by ``cu_q`` (query row offsets per document)
and ``q_pos`` (position, inside the document's keys, of each document's first
query).

Large tensors are drawn in row chunks of ``CHUNK_ELEMS`` elements so that the
float32 staging buffer stays small; the chunking is part of the definition.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

CHUNK_ELEMS = 1 << 26


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    D: int
    kpool: int
    index_topk: int
    tail: bool = True
    n_docs: int = 1
    doc_len_range: tuple | None = None   # (lo, hi) for seeded packed-THD lengths
    equal_docs: bool = False              # batch of equal sequences
    fp8: bool = False
    seed: int = 0
    queries: str = "all"                  # "all" | "last" | "chunk:N"
    desc: str = ""

    @property
    def Kp(self) -> int:
        return self.index_topk // self.kpool


WORKLOADS = {
    "tiny": Workload("tiny", T=256, H=4, D=32, kpool=4, index_topk=32,
                     desc="Tiny single sequence T=256 H=4 D=32 kpool=4 index_topk=32"),
    "single_8k": Workload("single_8k", T=8192, H=64, D=128, kpool=4, index_topk=2048,
                          desc="Single sequence T=8192 H=64 D=128 kpool=4 index_topk=2048"),
    "thd_32k": Workload("thd_32k", T=32768, H=64, D=128, kpool=4, index_topk=2048,
                        n_docs=16, doc_len_range=(256, 4096),
                        desc="Packed THD: 16 documents, lengths U[256,4096] rescaled to "
                             "32768 tokens, H=64 D=128 kpool=4 index_topk=2048"),
    "long_128k": Workload("long_128k", T=131072, H=64, D=128, kpool=4, index_topk=2048,
                          desc="Long single sequence T=131072 H=64 D=128 kpool=4 "
                               "index_topk=2048"),
    "fp8_2x32k": Workload("fp8_2x32k", T=65536, H=64, D=128, kpool=4, index_topk=2048,
                          n_docs=2, equal_docs=True, fp8=True,
                          desc="FP8 indexer mode: 2 sequences of 32768 tokens, H=64 D=128 "
                               "kpool=4 index_topk=2048, E4M3 scoring"),
    "fp8_128k": Workload("fp8_128k", T=131072, H=64, D=128, kpool=4, index_topk=2048, fp8=True,
                         desc="FP8 indexer mode at T=131072: one sequence, H=64 D=128 kpool=4 "
                              "index_topk=2048, E4M3 scoring"),
    "chunk_16k_of_128k": Workload("chunk_16k_of_128k", T=131072, H=64, D=128, kpool=4,
                                  index_topk=2048, queries="chunk:16384",
                                  desc="Chunked prefill: the last 16384-token chunk of a "
                                       "131072-token sequence (queries at positions "
                                       "114688..131071 over all 131072 keys), H=64 D=128 "
                                       "kpool=4 index_topk=2048"),
    "decode_128x32k": Workload("decode_128x32k", T=128 * 32768, H=64, D=128, kpool=4,
                               index_topk=2048, n_docs=128, doc_len_range=(8192, 57344),
                               queries="last",
                               desc="Decode: one query per sequence at its last key, 128 "
                                    "sequences with lengths U[8192,57344] rescaled to "
                                    "4194304 keys, H=64 D=128 kpool=4 index_topk=2048"),
}

# Key-path fusion (hidden states -> projected keys, k_norm, gate -> pooled keys):
# the hidden size is not given by the pages; 6144 is used for measurement.
PROJECTION_WORKLOADS = {
    "proj_128k": dict(T=131072, hidden=6144, D=128, kpool=4,
                      desc="Key path fused with compression: T=131072 hidden states of 6144, "
                           "D=128, kpool=4 (x ~ N(0,1), W ~ N(0,1/hidden) bf16)"),
}


# The sparse attention that consumes the selection (absorbed NoPE MLA): 64
# heads and a 512-wide latent (the pages' production config once the rotary
# slice is gone); the softmax scale is not given by the pages, 512^-0.5 is used.
MLA_HEADS = 64
MLA_DC = 512
MLA_SCALE = 512 ** -0.5
MLA_WORKLOADS = {
    "mla_32k": Workload("mla_32k", T=32768, H=64, D=128, kpool=4, index_topk=2048,
                        desc="Sparse attention over the indexer's selection: one sequence "
                             "T=32768, 64 heads, latent 512, kpool=4 index_topk=2048 with the "
                             "tail (up to 2051 tokens per query), fused expansion"),
    "mla_thd_32k": Workload("mla_thd_32k", T=32768, H=64, D=128, kpool=4, index_topk=2048,
                            n_docs=16, doc_len_range=(256, 4096),
                            desc="Sparse attention over the indexer's selection, packed THD: "
                                 "16 documents, lengths U[256,4096] rescaled to 32768 tokens, "
                                 "64 heads, latent 512, fused expansion"),
}


@dataclass
class MlaInputs:
    q: torch.Tensor      # bf16 [T, 64, 512] absorbed queries
    kv: torch.Tensor     # bf16 [Tk, 512] latent rows (keys and values)
    scale: float


def make_mla_inputs(T: int, Tk: int | None = None, seed: int = 0) -> MlaInputs:
    """q ~ N(0, 1) then kv ~ N(0, 1), both rounded to bfloat16 (one generator
    seeded with seed + 7919, q drawn first)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 7919)
    q = _normal_bf16((T, MLA_HEADS, MLA_DC), gen)
    kv = _normal_bf16((T if Tk is None else Tk, MLA_DC), gen)
    return MlaInputs(q, kv, MLA_SCALE)


def doc_lengths(wl: Workload, gen: torch.Generator) -> list:
    if wl.n_docs == 1:
        return [wl.T]
    if wl.equal_docs:
        assert wl.T % wl.n_docs == 0
        return [wl.T // wl.n_docs] * wl.n_docs
    lo, hi = wl.doc_len_range
    u = torch.rand(wl.n_docs, generator=gen, dtype=torch.float64) * (hi - lo) + lo
    lens = [int(math.floor(float(x) * wl.T / float(u.sum()))) for x in u]
    lens[-1] += wl.T - sum(lens)
    return lens


def _normal_bf16(shape, gen, scale=1.0):
    n = 1
    for s in shape:
        n *= s
    out = torch.empty(n, dtype=torch.bfloat16)
    pos = 0
    while pos < n:
        m = min(CHUNK_ELEMS, n - pos)
        x = torch.randn(m, generator=gen, dtype=torch.float32)
        if scale != 1.0:
            x *= scale
        out[pos:pos + m] = x.to(torch.bfloat16)
        pos += m
    return out.view(*shape)


def query_layout(queries: str, lens: list):
    """Per-document query counts and first positions of a positioned
    workload, or None for a prefill."""
    if queries == "all":
        return None
    if queries == "last":
        n = [1 if L > 0 else 0 for L in lens]
    elif queries.startswith("chunk:"):
        c = int(queries.split(":", 1)[1])
        n = [min(c, L) for L in lens]
    else:
        raise ValueError("unknown query layout %r" % queries)
    cu_q = [0]
    for x in n:
        cu_q.append(cu_q[-1] + x)
    q_pos = [L - x for L, x in zip(lens, n)]
    return cu_q, q_pos


@dataclass
class Inputs:
    wl: Workload
    cu_seqlens: torch.Tensor      # int32 [n_docs + 1] (key tokens)
    q: torch.Tensor               # bf16 [Tq, H, D]
    k: torch.Tensor               # bf16 [T, D]
    gate: torch.Tensor            # bf16 [T, D]
    ape: torch.Tensor             # fp32 [kpool, D]
    w: torch.Tensor               # fp32 [Tq, H]
    cu_q: torch.Tensor | None = None     # int32 [n_docs + 1], positioned workloads
    q_pos: torch.Tensor | None = None    # int32 [n_docs], positioned workloads
    extra: dict = field(default_factory=dict)

    @property
    def Tq(self) -> int:
        return self.q.shape[0]


def make_inputs(wl: Workload, seed: int | None = None, T: int | None = None) -> Inputs:
    """Draw the inputs of workload ``wl`` on the CPU.  ``T`` overrides the
    token count (same recipe, used for reduced-size parity cases)."""
    if T is not None and T != wl.T:
        from dataclasses import replace
        wl = replace(wl, T=T)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(wl.seed if seed is None else seed)
    lens = doc_lengths(wl, gen)
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    cu_seqlens = torch.tensor(cu, dtype=torch.int32)
    lay = query_layout(wl.queries, lens)
    Tq = wl.T if lay is None else lay[0][-1]
    q = _normal_bf16((Tq, wl.H, wl.D), gen)
    k = _normal_bf16((wl.T, wl.D), gen)
    gate = _normal_bf16((wl.T, wl.D), gen)
    ape = torch.randn(wl.kpool, wl.D, generator=gen, dtype=torch.float32) * 0.1
    w = torch.randn(Tq, wl.H, generator=gen, dtype=torch.float32) / math.sqrt(wl.H)
    if lay is None:
        return Inputs(wl, cu_seqlens, q, k, gate, ape, w)
    return Inputs(wl, cu_seqlens, q, k, gate, ape, w,
                  torch.tensor(lay[0], dtype=torch.int32), torch.tensor(lay[1], dtype=torch.int32))


@dataclass
class ProjectionInputs:
    """Inputs of the key path in front of compression (hidden states and the
    key / gate projection weights, k_norm's weight and bias)."""
    cu_seqlens: torch.Tensor      # int32 [n_docs + 1]
    x: torch.Tensor               # bf16 [T, hidden]
    w_kg: torch.Tensor            # bf16 [2D, hidden]: key projection rows, then gate rows
    gamma: torch.Tensor           # fp32 [D]
    beta: torch.Tensor            # fp32 [D]
    ape: torch.Tensor             # fp32 [kpool, D]
    eps: float = 1e-6


def make_projection_inputs(T: int, hidden: int, D: int, kpool: int, n_docs: int = 1,
                           doc_len_range=None, seed: int = 0) -> ProjectionInputs:
    """Draw order (seeded torch.Generator on the CPU): document lengths (as for
    packed-THD workloads), x ~ N(0, 1) and w_kg ~ N(0, 1/hidden) drawn in float32
    and rounded to bfloat16, gamma = 1 + N(0, 0.1^2), beta ~ N(0, 0.1^2),
    ape ~ N(0, 0.1^2)."""
    wl = Workload("proj", T=T, H=1, D=D, kpool=kpool, index_topk=kpool, n_docs=n_docs,
                  doc_len_range=doc_len_range)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    lens = doc_lengths(wl, gen)
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    x = _normal_bf16((T, hidden), gen)
    w_kg = _normal_bf16((2 * D, hidden), gen, scale=1.0 / math.sqrt(hidden))
    gamma = 1.0 + 0.1 * torch.randn(D, generator=gen, dtype=torch.float32)
    beta = 0.1 * torch.randn(D, generator=gen, dtype=torch.float32)
    ape = 0.1 * torch.randn(kpool, D, generator=gen, dtype=torch.float32)
    return ProjectionInputs(torch.tensor(cu, dtype=torch.int32), x, w_kg, gamma, beta, ape)


def sample_rows(T: int, n_sample: int = 1024, edge: int = 64, seed: int = 0,
                lo: int = 0, hi: int | None = None) -> torch.Tensor:
    """Rows checked at full size: ``n_sample`` rows drawn without replacement
    from [lo+edge, hi-edge) plus the first and last ``edge`` rows of
    [lo, hi).  Sorted, int64."""
    hi = T if hi is None else hi
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    inner = hi - lo - 2 * edge
    if inner <= n_sample:
        return torch.arange(lo, hi, dtype=torch.int64)
    pick = torch.randperm(inner, generator=gen)[:n_sample] + lo + edge
    rows = torch.cat([torch.arange(lo, lo + edge), pick, torch.arange(hi - edge, hi)])
    return torch.sort(rows.to(torch.int64)).values


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (a view, no arithmetic)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
