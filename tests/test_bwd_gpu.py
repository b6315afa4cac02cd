"""Backward parity on a GB300: dQ, dK, dV from the CUDA path (C ABI, using
the forward's own O and LSE) against the oracle's analytic fp64 gradients
on identical seeded bf16 inputs."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attn_ref
from tests.gpu_util import assert_close, assert_close_scaled, d_term_bounds, to64

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


@pytest.mark.parametrize("scale", [-0.088, 0.0])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 4, 2, 300, 300, 128), (1, 2, 2, 100, 400, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_any_finite_scale(fa, shape, causal, scale):
    """scale is any finite number: negative (the row max is taken over
    scale * s, not s) and zero (every visible key weighted equally)."""
    B, Hq, Hkv, Nq, Nk, d = shape
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=int(1000 * scale) % 997 + Nq, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    xs = [x[n].double().numpy() for n in ("q", "k", "v", "do")]
    ro, rlse = attn_ref.forward(*xs[:3], scale, causal)
    assert_close("o", to64(o), ro)
    fin = np.isfinite(rlse)
    glse = to64(lse)
    assert np.array_equal(np.isfinite(glse), fin)
    assert float(np.abs(glse[fin] - rlse[fin]).max(initial=0.0)) <= 1e-3
    rdq, rdk, rdv = attn_ref.backward(*xs, scale, causal)
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


def test_gqa_causal_full_size_one_group(fa):
    """GQA backward at scale: the causal GQA workload's shape (B=1, Hq=32,
    Hkv=8, N=16384) with the backward workload's input distribution (all
    N(0,1)), run whole on the GPU; the oracle recomputes every gradient of
    one kv group (kv head 5 and its query heads 20-23), dK and dV summed over
    the group. dV and dK of the first keys sum over all 4 x 16384 queries of
    the group and reach |x| of 4-8, where one bf16 ulp is 0.03 and output
    rounding alone costs up to 1.6e-2, so the elementwise bound grows with
    the value (assert_close_scaled); mean-abs stays at 2e-3."""
    w = workloads.WORKLOADS[3]
    x = workloads.make_inputs(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.seed, with_dout=True)
    dq, dk, dv = gpu_grads(fa, x, w.causal, w.scale)
    g = w.Hq // w.Hkv
    kvh = 5
    hs = slice(kvh * g, (kvh + 1) * g)
    qs, dos = (x[n][:, :, hs].double().numpy() for n in ("q", "do"))
    ks, vs = (x[n][:, :, kvh:kvh + 1].double().numpy() for n in ("k", "v"))
    rdq, rdk, rdv = attn_ref.backward(qs, ks, vs, dos, w.scale, w.causal)
    assert_close_scaled("dq[group 5]", to64(dq[:, :, hs]), rdq)
    assert_close_scaled("dk[kv 5]", to64(dk[:, :, kvh:kvh + 1]), rdk)
    assert_close_scaled("dv[kv 5]", to64(dv[:, :, kvh:kvh + 1]), rdv)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()


def test_gqa_causal_workload_distribution_one_group(fa):
    """The backward of the causal GQA workload itself, as the benchmark step
    runs it: B=1, Hq=32, Hkv=8, N=16384, Q and K ~ N(0, 2^2), V ~ N(0, 1),
    dO ~ N(0, 1) drawn after them from the workload's seed, O and LSE from
    the GPU forward. Every gradient of one kv group (kv head 2, query heads
    8-11) against the oracle.

    With logits of standard deviation 4 the rows are nearly one-hot; dK and
    dV reach |x| of 16-20, where one bf16 ulp is 0.125: the rounding of the
    output alone exceeds the fixed max-abs 2e-2 for hundreds of elements, so
    that bound cannot hold for a bf16-output backward at this distribution.
    Elementwise bound used, each term from the arithmetic:
      2e-2                the published tolerance (fp32 accumulation etc.)
      + 2^-8 |ref|        rounding the output to bf16 (half an ulp)
      + 2^-8 a            rounding P (dV) and dS (dQ, dK) to bf16 before the
                          GEMMs; a = the oracle's backward_abs_terms
                          (scale sum |dS| |K| and so on), which the
                          cancellation in dS = P (dP - D) can make much
                          larger than |ref|
      + the D term        D_i is formed from the bf16 O the backward takes
                          as input (d_term_bounds): up to scale |dD| P|K|
                          for dQ and scale P^T(|dD| |Q|) for dK
    and mean-abs 2e-3 as for the published workloads."""
    w = workloads.WORKLOADS[3]
    x = workloads.workload_inputs(w, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    g = w.Hq // w.Hkv
    kvh = 2
    hs = slice(kvh * g, (kvh + 1) * g)
    qs, dos = (x[n][:, :, hs].double().numpy() for n in ("q", "do"))
    ks, vs = (x[n][:, :, kvh:kvh + 1].double().numpy() for n in ("k", "v"))
    rdq, rdk, rdv = attn_ref.backward(qs, ks, vs, dos, w.scale, w.causal)
    a_dq, a_dk, a_dv = attn_ref.backward_abs_terms(qs, ks, vs, dos, w.scale, w.causal)
    ro, _ = attn_ref.forward(qs, ks, vs, w.scale, w.causal)
    bdq, bdk = d_term_bounds(qs, ks, dos, to64(o[:, :, hs]), ro, w.scale, w.causal)
    for name, got, ref, extra in (("dq[group 2]", dq[:, :, hs], rdq, 2.0 ** -8 * a_dq + bdq),
                                  ("dk[kv 2]", dk[:, :, kvh:kvh + 1], rdk, 2.0 ** -8 * a_dk + bdk),
                                  ("dv[kv 2]", dv[:, :, kvh:kvh + 1], rdv, 2.0 ** -8 * a_dv)):
        assert_close_scaled(name, to64(got), ref, rel=2.0 ** -8, extra=extra)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()


@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths_at_scale(fa, causal):
    """Nq != Nk, neither a multiple of 128, GQA, both passes, every element
    against the oracle (bottom-right causal alignment: the first
    Nk - Nq keys are visible to every row)."""
    B, Hq, Hkv, Nq, Nk, d = 1, 8, 2, 3000, 5000, 128
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=24 + int(causal), with_dout=True)
    scale = d ** -0.5
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    ro, rlse = attn_ref.forward(*(x[n].double().numpy() for n in ("q", "k", "v")), scale, causal)
    assert_close("o", to64(o), ro)
    assert_close("lse", to64(lse), rlse, max_tol=1e-3, mean_tol=1e-3)
    dq, dk, dv = gpu_grads(fa, x, causal, scale)
    rdq, rdk, rdv = attn_ref.backward(*(x[n].double().numpy() for n in ("q", "k", "v", "do")), scale, causal)
    assert_close("dq", to64(dq), rdq)
    assert_close("dk", to64(dk), rdk)
    assert_close("dv", to64(dv), rdv)


BWD_WINDOWS = [
    # B, Hq, Hkv, Nq, Nk, d, (left, right)
    (1, 2, 2, 300, 300, 128, (64, 0)),
    (1, 2, 1, 700, 700, 64, (200, 0)),
    (1, 2, 2, 513, 513, 128, (128, 128)),
    (1, 2, 2, 400, 900, 128, (300, 50)),    # Nq < Nk
    (1, 2, 2, 900, 400, 128, (100, 0)),     # Nq > Nk: rows with no visible key
    (1, 2, 2, 600, 600, 64, (-1, 300)),     # right bound only
    (1, 3, 3, 1000, 1000, 128, (500, -1)),  # left bound only
    (2, 4, 2, 1024, 1024, 128, (0, 0)),     # one key per row (GQA)
]


@pytest.mark.parametrize("shape", BWD_WINDOWS, ids=lambda s: "x".join(map(str, s[:6])) + f"-w{s[6][0]}_{s[6][1]}")
def test_window(fa, shape):
    B, Hq, Hkv, Nq, Nk, d, window = shape
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape[:6]) + 3 * window[0] + window[1], with_dout=True)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, scale=scale, window=window)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, scale=scale, window=window)
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    rdq, rdk, rdv = attn_ref.backward(*(x[n].double().numpy() for n in ("q", "k", "v", "do")), scale, False,
                                      window=window)
    assert_close("dq", to64(dq), rdq)
    assert_close("dk", to64(dk), rdk)
    assert_close("dv", to64(dv), rdv)


def test_window_full_size_sampled_heads(fa):
    """A causal local window of 1024 keys at N = 8192 (B=1, H=8): every
    gradient of two heads against the oracle."""
    B, H, N, d, window = 1, 8, 8192, 128, (1023, 0)
    x = workloads.make_inputs(B, H, H, N, N, d, seed=43, with_dout=True)
    scale = d ** -0.5
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, scale=scale, window=window)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, scale=scale, window=window)
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    for h in (0, 5):
        sl = lambda t: t[:, :, h:h + 1].double().numpy()
        rdq, rdk, rdv = attn_ref.backward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["do"]), scale, False, window=window)
        assert_close(f"dq[h{h}]", to64(dq[:, :, h:h + 1]), rdq)
        assert_close(f"dk[h{h}]", to64(dk[:, :, h:h + 1]), rdk)
        assert_close(f"dv[h{h}]", to64(dv[:, :, h:h + 1]), rdv)


# The causal backward's split of its last round (fa_tune FA_TUNE_BWD_SPLIT
# forces the count m of pairs per kv head that run as single tiles): with
# GQA at d = 128 each single is split once more per query head, whose dK/dV
# are partial sums kept in fp32 and summed by a last pass; otherwise
# the singles take the whole group. Small shapes, forced m, against the
# oracle element by element.
SPLITS = [
    # B, Hq, Hkv, Nq, Nk, d, m
    (2, 8, 2, 1000, 1000, 128, 1),   # 8 key tiles, group 4: pieces per query head
    (2, 8, 2, 1000, 1000, 128, 4),   # every pair split
    (1, 4, 2, 1100, 1100, 128, 2),   # 9 key tiles: the middle tile is a tail tile too
    (1, 4, 2, 1100, 1100, 128, 0),   # only the middle tile
    (1, 6, 3, 600, 1000, 128, 2),    # Nq < Nk
    (1, 4, 4, 900, 900, 128, 3),     # MHA: singles take the whole (one-head) group
    (1, 4, 2, 700, 700, 64, 2),      # d = 64: singles take the whole group
]


@pytest.mark.parametrize("shape", SPLITS, ids=lambda s: "x".join(map(str, s)))
def test_forced_split_matches_oracle(fa, shape):
    B, Hq, Hkv, Nq, Nk, d, m = shape
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape) + 7, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    assert fa.fa_tune(fa.TUNE_BWD_SPLIT, m) == 0
    try:
        dq, dk, dv = gpu_grads(fa, x, True, scale)
    finally:
        fa.fa_tune(fa.TUNE_BWD_SPLIT, -1)
    rdq, rdk, rdv = attn_ref.backward(*(x[n].double().numpy() for n in ("q", "k", "v", "do")), scale, True)
    assert_close("dq", to64(dq), rdq)
    # GQA dK/dV sum over the group's queries and pass |x| = 4, where output
    # rounding alone can exceed 2e-2: the bound grows with the value
    assert_close_scaled("dk", to64(dk), rdk)
    assert_close_scaled("dv", to64(dv), rdv)


def test_forced_split_agrees_with_model_split(fa):
    """The same inputs with the split count from the model and with every
    pair split into pieces: the gradients agree within the fp32 summation
    order (dK/dV of a tile summed in TMEM over its heads, or in fp32 over
    its pieces) and one bf16 rounding; and a second run with pieces gives
    the same dK, dV bit for bit (the pieces are summed in a fixed order)."""
    B, Hq, Hkv, N, d = 1, 8, 2, 1536, 128
    x = workloads.make_inputs(B, Hq, Hkv, N, N, d, seed=91, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    ref = gpu_grads(fa, x, True, scale)
    assert fa.fa_tune(fa.TUNE_BWD_SPLIT, 6) == 0
    try:
        got = gpu_grads(fa, x, True, scale)
        again = gpu_grads(fa, x, True, scale)
    finally:
        fa.fa_tune(fa.TUNE_BWD_SPLIT, -1)
    assert torch.equal(got[1], again[1]) and torch.equal(got[2], again[2])
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        a64, b64 = a.double(), b.double()
        ulp = torch.maximum(a64.abs(), b64.abs()) * 2.0 ** -7 + 1e-6
        assert ((a64 - b64).abs() <= ulp).all(), (name, (a64 - b64).abs().max().item())
