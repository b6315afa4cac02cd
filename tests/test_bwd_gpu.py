"""Backward parity on a GB300: dQ, dK, dV from the CUDA path (C ABI, using
the forward's own O and LSE) against the oracle's analytic fp64 gradients
on identical seeded bf16 inputs."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attn_ref
from tests.gpu_util import assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_99_gb300 as m
    m.fa_debug_set(0, 0)
    return m


def gpu_grads(fa, x, causal, scale):
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    return dq, dk, dv


SMALL = [
    # B, Hq, Hkv, Nq, Nk, d
    (1, 1, 1, 1, 1, 128),
    (1, 2, 2, 17, 17, 64),
    (1, 2, 1, 128, 128, 128),
    (2, 2, 2, 129, 129, 64),
    (1, 4, 2, 255, 255, 128),
    (1, 2, 2, 256, 256, 128),
    (1, 3, 1, 300, 300, 128),
    (1, 2, 2, 100, 400, 128),   # Nq < Nk
    (1, 2, 2, 400, 100, 64),    # Nq > Nk: causal rows with no visible key
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(fa, shape, causal):
    B, Hq, Hkv, Nq, Nk, d = shape
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=hash((shape, causal)) % 10000, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = gpu_grads(fa, x, causal, scale)
    rdq, rdk, rdv = attn_ref.backward(*(x[n].double().numpy() for n in ("q", "k", "v", "do")), scale, causal)
    assert_close("dq", to64(dq), rdq)
    assert_close("dk", to64(dk), rdk)
    assert_close("dv", to64(dv), rdv)


def test_workload_full_size_sampled_heads(fa):
    """Full-size backward workload (the benchmark's launch configuration);
    the oracle recomputes every gradient of a few (batch, head) slices."""
    w = workloads.WORKLOADS[4]
    x = workloads.workload_inputs(w)
    dq, dk, dv = gpu_grads(fa, x, w.causal, w.scale)
    gdq, gdk, gdv = to64(dq), to64(dk), to64(dv)
    for b, h in [(0, 0), (w.B - 1, w.Hq - 1), (1, 7)]:
        sl = lambda t: t[b:b + 1, :, h:h + 1].double().numpy()
        rdq, rdk, rdv = attn_ref.backward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["do"]), w.scale, w.causal)
        assert_close(f"dq[b{b},h{h}]", gdq[b:b + 1, :, h:h + 1], rdq)
        assert_close(f"dk[b{b},h{h}]", gdk[b:b + 1, :, h:h + 1], rdk)
        assert_close(f"dv[b{b},h{h}]", gdv[b:b + 1, :, h:h + 1], rdv)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()


def test_gqa_grads_group_sum(fa):
    B, Hq, Hkv, N, d = 1, 8, 2, 384, 128
    x = workloads.make_inputs(B, Hq, Hkv, N, N, d, seed=21, with_dout=True)
    scale = d ** -0.5
    dq, dk, dv = gpu_grads(fa, x, True, scale)
    rdq, rdk, rdv = attn_ref.backward(*(x[n].double().numpy() for n in ("q", "k", "v", "do")), scale, True)
    assert_close("dq", to64(dq), rdq)
    assert_close("dk", to64(dk), rdk)
    assert_close("dv", to64(dv), rdv)


def test_dk_dv_deterministic(fa):
    B, H, N, d = 2, 4, 512, 128
    x = workloads.make_inputs(B, H, H, N, N, d, seed=22, with_dout=True)
    a = gpu_grads(fa, x, True, d ** -0.5)
    b = gpu_grads(fa, x, True, d ** -0.5)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2e-2  # dQ sums in arbitrary order


def test_gradient_identities_on_gpu(fa):
    # sum over keys of dV = sum over queries of dO (rows of P sum to 1);
    # sum over keys of dK = 0 (rows of dS sum to 0)
    B, H, N, d = 1, 2, 640, 128
    x = workloads.make_inputs(B, H, H, N, N, d, seed=23, with_dout=True)
    dq, dk, dv = gpu_grads(fa, x, True, d ** -0.5)
    want = x["do"].double().sum(dim=1)
    assert (dv.double().cpu().sum(dim=1) - want).abs().max().item() <= 0.5
    assert dk.double().cpu().sum(dim=1).abs().max().item() <= 0.5
