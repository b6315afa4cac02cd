"""The forward's exp2 split on a GB300 (fa_tune FA_TUNE_EXP2_SPLIT): with one
column pair in every N of the softmax's exponentials evaluated by the fitted
polynomial on the FMA pipes (N = 1: all of them), the bf16 and e4m3 forwards
still match the oracle, and differ from the all-special-function-unit kernels
only by the polynomial's rounding.

The split follows the FlashAttention-4 article on smntcn.com (part of the
exponentials emulated in software on the FMA pipes)."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attn_ref
from tests.gpu_util import assert_close, assert_lse, to64

pytestmark = pytest.mark.gpu

SPLITS = [1, 2, 4, 8]


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_99_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    m.fa_debug_set(0, 0)
    assert m.fa_tune(m.TUNE_EXP2_SPLIT, 0) == 0
    yield m
    m.fa_tune(m.TUNE_EXP2_SPLIT, 0)


def forward_with_split(fa, x, causal, scale, split):
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    assert fa.fa_tune(fa.TUNE_EXP2_SPLIT, split) == 0
    try:
        o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
        torch.cuda.synchronize()
    finally:
        fa.fa_tune(fa.TUNE_EXP2_SPLIT, 0)
    assert fa.fa_get_status() == 0
    return o, lse


SHAPES = [
    # B, Hq, Hkv, Nq, Nk, d
    (1, 2, 1, 17, 17, 128),
    (1, 4, 2, 300, 300, 128),
    (2, 2, 2, 513, 513, 64),
    (1, 2, 2, 100, 700, 128),   # Nq < Nk
    (1, 2, 2, 700, 100, 128),   # Nq > Nk: causal rows with no visible key
]


@pytest.mark.parametrize("split", SPLITS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_split_matches_oracle(fa, shape, causal, split):
    B, Hq, Hkv, Nq, Nk, d = shape
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape) + 13 * split + causal)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_with_split(fa, x, causal, scale, split)
    ro, rlse = attn_ref.forward(*(x[n].double().numpy() for n in ("q", "k", "v")), scale, causal)
    assert_close("o", to64(o), ro)
    assert_lse(to64(lse), rlse)


@pytest.mark.parametrize("split", SPLITS)
def test_split_differs_only_by_polynomial_rounding(fa, split):
    """Against the all-special-function-unit kernel on the same inputs (Q, K
    with σ = 2, so many probabilities are far from 1). Each exponential moves
    by at most the polynomial's relative error (7.5e-5) plus ex2.approx's
    (2^-22), in the numerator P V and in the row sum l alike (2 x 7.5e-5);
    the bf16 rounding of P before the P V GEMM can then flip by one bf16 ulp
    (at most 2^-7 of the value). So, with S_ic = sum_j P_ij |V_jc| (the
    oracle's attention of |V|): |dO_ic| <= (1.5e-4 + 2^-7) S_ic + one bf16
    ulp of O, and LSE moves by at most about 1e-4 (l sums the fp32
    probabilities)."""
    B, H, N, d = 1, 4, 640, 128
    x = workloads.make_inputs(B, H, H, N, N, d, seed=91 + split, sigma_qk=2.0)
    scale = 1.0 / math.sqrt(d)
    qn, kn, vn = (x[n].double().numpy() for n in ("q", "k", "v"))
    for causal in (False, True):
        o0, l0 = forward_with_split(fa, x, causal, scale, 0)
        o1, l1 = forward_with_split(fa, x, causal, scale, split)
        dl = (l1.double() - l0.double()).abs().max().item()
        assert dl <= 1e-4, (causal, dl)
        s_abs, _ = attn_ref.forward(qn, kn, np.abs(vn), scale, causal)
        a0, a1 = to64(o0), to64(o1)
        ulp = np.maximum(np.abs(a0), np.abs(a1)) * 2.0 ** -7
        bound = (1.5e-4 + 2.0 ** -7) * s_abs + ulp + 1e-6
        diff = np.abs(a1 - a0)
        assert (diff <= bound).all(), (causal, float((diff - bound).max()))
        assert float(diff.mean()) <= 1e-3, (causal, float(diff.mean()))


@pytest.mark.parametrize("split", [2, 8])
def test_split_causal_workload_whole_head(fa, split):
    """The causal B=2, H=16, N=8192 workload with the split on: every row of
    the last head of the last batch element against the oracle."""
    w = workloads.WORKLOADS[2]
    x = workloads.workload_inputs(w)
    o, lse = forward_with_split(fa, x, w.causal, w.scale, split)
    b, h = w.B - 1, w.Hq - 1
    sl = lambda t: t[b:b + 1, :, h:h + 1].double().numpy()
    ro, rlse = attn_ref.forward(sl(x["q"]), sl(x["k"]), sl(x["v"]), w.scale, w.causal)
    assert_close(f"o[b{b},h{h}]", to64(o[b:b + 1, :, h:h + 1]), ro)
    assert_lse(to64(lse[b:b + 1, h:h + 1]), rlse)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("split", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_split_fp8_against_default(fa, causal, split):
    """The e4m3 forward with the split on: against the same call without it.
    The codes of Q, K and V are the same; P's e4m3 rounding can flip where
    the polynomial moves a probability across a rounding boundary (one e4m3
    ulp, 2^-3 relative, of that P), so O moves by at most 2^-3 of one P_ij
    |V_j| per flipped code plus the polynomial's relative error; LSE by the
    polynomial's relative error only (l sums the fp32 probabilities)."""
    B, Hq, Hkv, N, d = 1, 4, 2, 300, 128
    x = workloads.make_inputs(B, Hq, Hkv, N, N, d, seed=55 + causal + split)
    scale = 1.0 / math.sqrt(d)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o0, l0 = fa.forward_fp8(q, k, v, causal=causal, scale=scale)
    assert fa.fa_tune(fa.TUNE_EXP2_SPLIT, split) == 0
    try:
        o1, l1 = fa.forward_fp8(q, k, v, causal=causal, scale=scale)
        torch.cuda.synchronize()
    finally:
        fa.fa_tune(fa.TUNE_EXP2_SPLIT, 0)
    assert fa.fa_get_status() == 0
    g0, g1 = to64(l0), to64(l1)
    fin = np.isfinite(g0)
    assert np.array_equal(fin, np.isfinite(g1))
    assert float(np.abs(g1[fin] - g0[fin]).max(initial=0.0)) <= 1e-4
    d_o = np.abs(to64(o1) - to64(o0))
    vmax = float(x["v"].double().abs().max())
    assert float(d_o.max()) <= 2.0 ** -3 * vmax + 2e-3, float(d_o.max())
    assert float(d_o.mean()) <= 2e-3, float(d_o.mean())
