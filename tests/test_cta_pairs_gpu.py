"""The d = 128 forward on pairs of CTAs (fa_tune FA_TUNE_CTA_PAIRS = 1): a
cluster of two CTAs takes 512 query rows at a time and the even CTA issues
tcgen05.mma with cta_group::2 (M = 256 over both CTAs' tensor memory), each
CTA loading half of every K and V tile. Checked against the fp64 oracle on
small, ragged, grouped-query and masked shapes, the row-split tail, whole
heads of the full-size d = 128 workloads, and against the one-CTA kernel.

The pairs follow the FlashAttention-4 article on smntcn.com (fifth-generation
tensor cores with 256 KB of tensor memory per SM; larger MMA tiles)."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attn_ref
from tests.gpu_util import assert_close, assert_lse, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_99_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    m.fa_debug_set(0, 0)
    assert m.fa_tune(m.TUNE_CTA_PAIRS, 0) == 0
    yield m
    m.fa_tune(m.TUNE_CTA_PAIRS, 0)


def paired_forward(fa, q, k, v, causal, scale):
    assert fa.fa_tune(fa.TUNE_CTA_PAIRS, 1) == 0
    try:
        o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
        torch.cuda.synchronize()
    finally:
        fa.fa_tune(fa.TUNE_CTA_PAIRS, 0)
    assert fa.fa_get_status() == 0
    return o, lse


SHAPES = [
    # B, Hq, Hkv, Nq, Nk
    (1, 2, 1, 17, 17),
    (1, 2, 2, 128, 128),
    (1, 4, 2, 300, 300),
    (2, 2, 2, 512, 512),
    (1, 2, 2, 513, 513),      # one row into a second 512-row unit
    (1, 4, 1, 1000, 1000),
    (1, 2, 2, 100, 700),      # Nq < Nk
    (1, 2, 2, 700, 100),      # Nq > Nk: causal rows with no visible key
    (1, 40, 40, 700, 384),    # 80 units over 76 pairs: row-split tail
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_pairs_match_oracle(fa, shape, causal):
    B, Hq, Hkv, Nq, Nk = shape
    d = 128
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape) + 3 * causal + 17)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    o, lse = paired_forward(fa, q, k, v, causal, scale)
    ro, rlse = attn_ref.forward(*(x[n].double().numpy() for n in ("q", "k", "v")), scale, causal)
    assert_close("o", to64(o), ro)
    assert_lse(to64(lse), rlse)


@pytest.mark.parametrize("scale", [-0.088, 0.0])
def test_pairs_any_finite_scale(fa, scale):
    B, Hq, Hkv, N, d = 1, 4, 2, 300, 128
    x = workloads.make_inputs(B, Hq, Hkv, N, N, d, seed=int(1000 * scale) % 997 + 5)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    for causal in (False, True):
        o, lse = paired_forward(fa, q, k, v, causal, scale)
        ro, rlse = attn_ref.forward(*(x[n].double().numpy() for n in ("q", "k", "v")), scale, causal)
        assert_close("o", to64(o), ro)
        assert_lse(to64(lse), rlse)


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_pairs_workload_whole_heads(fa, idx):
    """The full-size d = 128 forward workloads on CTA pairs: every row of the
    first and the last (batch, head), and finite everywhere."""
    w = workloads.WORKLOADS[idx]
    x = workloads.workload_inputs(w)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = paired_forward(fa, q, k, v, w.causal, w.scale)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    go, glse = to64(o), to64(lse)
    for b, h in ((0, 0), (w.B - 1, w.Hq - 1)):
        kv = h // (w.Hq // w.Hkv)
        sl = lambda t, hh: t[b:b + 1, :, hh:hh + 1].double().numpy()
        ro, rlse = attn_ref.forward(sl(x["q"], h), sl(x["k"], kv), sl(x["v"], kv), w.scale, w.causal)
        assert_close(f"o[b{b},h{h}]", go[b:b + 1, :, h:h + 1], ro)
        assert_lse(glse[b:b + 1, h:h + 1], rlse)


def test_pairs_agree_with_one_cta_kernel(fa):
    """Same inputs through both kernels: the GEMMs are the same products in
    the same K order, so O and LSE agree to a bf16 ulp (any difference comes
    from the order in which the tensor cores sum)."""
    B, Hq, Hkv, N, d = 2, 8, 2, 1536, 128
    x = workloads.make_inputs(B, Hq, Hkv, N, N, d, seed=77, sigma_qk=2.0)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    for causal in (False, True):
        o1, l1 = fa.forward(q, k, v, causal=causal)
        o2, l2 = paired_forward(fa, q, k, v, causal, 1.0 / math.sqrt(d))
        a1, a2 = o1.double(), o2.double()
        ulp = torch.maximum(a1.abs(), a2.abs()) * 2.0 ** -7 + 1e-6
        assert ((a1 - a2).abs() <= ulp).all(), (causal, (a1 - a2).abs().max().item())
        assert (l1.double() - l2.double()).abs().max().item() <= 1e-5


def test_pairs_knob_validates(fa):
    assert fa.fa_tune(fa.TUNE_CTA_PAIRS, 2) == 1
    assert fa.fa_tune(fa.TUNE_CTA_PAIRS, -1) == 1
    assert fa.fa_tune(fa.TUNE_CTA_PAIRS, 0) == 0
