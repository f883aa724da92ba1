"""kpool_project_compress: hidden states -> key and gate projections ->
k_norm -> pool compression in one tcgen05 kernel.

* Bit for bit against kpool_compress on the kernel's own rounded keys and
  gate (the fused epilogue pools in kpool_compress's operation order).
* Against the oracle's key path (exact projection, LayerNorm in double, each
  rounded once to BF16), with the allowances FP32 evaluation implies where a
  dot product or the normalisation cancels (see test_fused_matches_oracle).
* Operands on a coarse grid make the FP32 accumulation exact: the projected
  gate then equals the oracle's bit for bit and the keys are within 1 ulp plus
  the normalisation's FP32 allowance."""
import numpy as np
import pytest
import torch

from sparse_attention_kpool_compress_gb300 import workloads as W
from kpool_checks import bf16_bits, bf16_ulp_distance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_kpool_compress_gb300 as K
    return K


def _run(K, pi, kp):
    dev = torch.device("cuda")
    multi = pi.cu_seqlens.numel() > 2
    T = pi.x.shape[0]
    cu = cp = P = None
    if multi:
        cp_h, P = K.kpool_num_pools(pi.cu_seqlens, T, kp)
        cu, cp = pi.cu_seqlens.to(dev), cp_h.to(dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    pk, k, g = K.kpool_project_compress(pi.x.to(dev), pi.w_kg.to(dev), pi.gamma.to(dev),
                                        pi.beta.to(dev), pi.eps, pi.ape.to(dev), kp, cu, cp, P,
                                        want_k_gate=True, workspace=ws)
    ref = K.kpool_compress(k, g, pi.ape.to(dev), kp, cu, cp, P)
    torch.cuda.synchronize()
    assert K.kpool_read_status(ws) == 0
    return pk, k, g, ref


@pytest.mark.parametrize("T,hidden,kp,docs", [(512, 64, 4, None), (1000, 256, 4, None),
                                              (4096, 2048, 4, None), (700, 128, 1, None),
                                              (640, 128, 2, None), (1024, 192, 8, None),
                                              (2048, 64, 16, None), (2048, 64, 32, None),
                                              (3000, 512, 4, (5, (10, 1200)))])
def test_fused_equals_compress_of_its_own_keys(K, T, hidden, kp, docs):
    n_docs, rng = docs if docs else (1, None)
    pi = W.make_projection_inputs(T, hidden, 128, kp, n_docs, rng, seed=T + hidden + kp)
    pk, _, _, ref = _run(K, pi, kp)
    assert torch.equal(pk, ref)


def _ulp(exact):
    e = np.floor(np.log2(np.maximum(np.abs(exact), 2.0 ** -133)))
    return 2.0 ** (np.maximum(e, -126) - 7)


@pytest.mark.parametrize("T,hidden,kp,docs", [(1024, 1024, 4, None),
                                              (2500, 512, 4, (7, (1, 800))),
                                              (512, 6144, 4, None)])
def test_fused_matches_oracle(K, ora, T, hidden, kp, docs):
    """Projected gate and normalised keys against the oracle's key path, with
    the allowances that FP32 evaluation implies:
    * gate: within 1 ulp plus 2^-14 * sum_i |x_i w_i| (FP32 accumulation over
      `hidden` products; where the dot product cancels, its error is relative
      to that sum, not to the result);
    * keys: the FP32 accumulation of a projected key may land on the other
      side of a BF16 midpoint, so each projected key may be the oracle's or
      its BF16 neighbour; the bound is 1 ulp plus 2^-20 times the
      normalisation's condition scale plus one BF16 ulp of every projected key
      carried through the normalisation to first order (through the key
      itself, the mean and the variance).
    The fused pooled keys equal kpool_compress on the kernel's own keys and
    gate bit for bit (checked above), and kpool_compress holds the 1-ulp bar
    against the oracle on the same inputs (test_gpu_parity), which closes the
    chain; here the pooled keys are also compared end to end."""
    n_docs, rng = docs if docs else (1, None)
    pi = W.make_projection_inputs(T, hidden, 128, kp, n_docs, rng, seed=3 * T + hidden)
    pk, k, g, _ = _run(K, pi, kp)
    kb, gb, kp_ex, k_ex, g_ex, k_cond = ora.project_keys(W.bits(pi.x), W.bits(pi.w_kg),
                                                         pi.gamma.numpy(), pi.beta.numpy(),
                                                         pi.eps, want_exact=True)
    kv = k.float().cpu().numpy().astype(np.float64)
    gv = g.float().cpu().numpy().astype(np.float64)
    xd = np.abs(pi.x.double().numpy())
    wd = np.abs(pi.w_kg.double().numpy())
    g_cond = xd @ wd[128:].T
    g_err = np.abs(gv - g_ex)
    assert np.all(g_err <= _ulp(g_ex) + 2.0 ** -14 * g_cond), float((g_err / g_cond).max())
    # first-order bound of the keys with every projected key off by one BF16 ulp
    xr = np.asarray(torch.from_numpy(kp_ex).float().to(torch.bfloat16).double())
    u = _ulp(xr)
    mu = xr.mean(axis=1, keepdims=True)
    dev_ = np.abs(xr - mu)
    rs = 1.0 / np.sqrt((dev_ ** 2).mean(axis=1, keepdims=True) + pi.eps)
    ubar = u.mean(axis=1, keepdims=True)
    dvar = 2.0 * (dev_ * (u + ubar)).mean(axis=1, keepdims=True)
    gam = np.abs(pi.gamma.double().numpy())[None, :]
    carry = gam * ((u + ubar) * rs + dev_ * 0.5 * rs ** 3 * dvar)
    k_err = np.abs(kv - k_ex)
    tight = k_err <= _ulp(k_ex) + 2.0 ** -20 * k_cond
    print("gate: %.2e of elements differ from the oracle's rounding; keys: %.2e past 1 ulp "
          "(+ FP32 allowance)" % ((bf16_ulp_distance(bf16_bits(g), gb) > 0).mean(),
                                  (~tight).mean()))
    assert np.all(k_err <= _ulp(k_ex) + 2.0 ** -20 * k_cond + 1.1 * carry)
    cu = pi.cu_seqlens.numpy() if n_docs > 1 else None
    pkb, exact, cond = ora.compress(kb, gb, pi.ape.numpy(), cu, kp, want_cond=True)
    got = pk.float().cpu().numpy().astype(np.float64)
    assert got.shape == exact.shape
    pk_err = np.abs(got - exact)
    ok = pk_err <= _ulp(exact) + 2.0 ** -20 * cond
    print("pooled keys: %.2e of elements past 1 ulp (+ FP32 allowance) end to end" % (~ok).mean())
    assert (~ok).mean() <= 1e-2
    assert np.all(pk_err <= 4 * _ulp(exact) + 2.0 ** -7 * cond)


def test_grid_operands_project_exactly(K, ora):
    """x and weights on coarse grids (x in {-2..2}/8, w in {-2..2}/16): every
    product is a multiple of 2^-7 and every partial sum is exact in FP32, so the
    projected gate equals the oracle's bit for bit."""
    T, hidden, kp = 512, 2048, 4
    g = torch.Generator().manual_seed(5)
    pi = W.make_projection_inputs(T, hidden, 128, kp, seed=9)
    pi.x = (torch.randint(-2, 3, (T, hidden), generator=g).float() / 8).to(torch.bfloat16)
    pi.w_kg = (torch.randint(-2, 3, (256, hidden), generator=g).float() / 16).to(torch.bfloat16)
    _, k, gt, _ = _run(K, pi, kp)
    kb, gb, _, k_ex, _, k_cond = ora.project_keys(W.bits(pi.x), W.bits(pi.w_kg), pi.gamma.numpy(),
                                                  pi.beta.numpy(), pi.eps, want_exact=True)
    assert np.array_equal(bf16_bits(gt), gb)
    kv = k.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(kv - k_ex) <= _ulp(k_ex) + 2.0 ** -20 * k_cond)
