"""FP8 (e4m3) forward on a GB300 against the FP8 oracle: the attention of
the dequantised e4m3 tensors (oracle/attn_fp8_ref.py), elementwise within
the bound that rounding P to e4m3 allows, plus the incoherent transform's
effect on inputs with outlier channels."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attn_fp8_ref as f8
from oracle import attn_ref
from tests.gpu_util import to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_99_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    m.fa_debug_set(0, 0)
    return m


def fp8_case(fa, x, causal, incoherent, scale):
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward_fp8(q, k, v, causal=causal, scale=scale, incoherent=incoherent)
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    return to64(o), to64(lse)


def rounding_sd(qd, kd, vd, scale, causal):
    """Standard deviation of O's error if every P_ij is rounded to e4m3 with
    an independent error uniform in +-half an ulp (2^-4 relative):
    (2^-4 / sqrt(3)) * sqrt(sum_j P_ij^2 V_jc^2), per output element."""
    B, Nq, Hq, d = qd.shape
    g = Hq // kd.shape[2]
    out = np.zeros_like(qd)
    for b in range(B):
        for h in range(Hq):
            P = attn_ref.probabilities(qd[b, :, h], kd[b, :, h // g], scale, causal)
            out[b, :, h] = np.sqrt((P ** 2) @ (vd[b, :, h // g] ** 2))
    return 2.0 ** -4 / np.sqrt(3.0) * out


def near_tie(u, w):
    """Where |u| (code units, at most 448) lies within w of the midpoint
    between two neighbouring e4m3 values, and the spacing there."""
    a = np.abs(u)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -30)))
    step = np.exp2(np.maximum(e, -6.0) - 3.0)  # 3 mantissa bits; subnormal spacing below 2^-6
    frac = a / step - np.floor(a / step)
    return np.abs(frac - 0.5) * step <= w, step


def flip_terms(qn, kn, vd, qd, kd, scale, causal, incoherent):
    """Bounds on what e4m3 codes that differ between the GPU and the oracle
    can do. Without the transform there are none: x / s is exact for a
    power-of-two s, so both sides round the same value. With it the GPU
    forms Q M and K M in fp32: a butterfly of seven add/subtract levels, each
    rounding once (level-l partial sums feeding one output add up to at most
    ||x||_1 <= sqrt(128) ||x||_2 in magnitude), then one multiply by the fp32
    value of 2^-e / sqrt(128); in code units u (||u||_2 = ||x||_2 / s) its
    error is below 7 2^-24 ||u||_2 + 2^-23 |u| < 2^-21 ||u||_2 + 2^-23 |u|.
    So an element can round to the other neighbour only where its exact
    value lies that close to a tie (near_tie): the code then moves by one
    e4m3 step. With f = scale sq sk, a flip of q_ic moves S_ij by at
    most f step kmax_c (kmax_c = max_j |k8_jc|) and a flip of k_jc by at most
    f |q8_ic| step, so
        |dS_ij| <= f (dq_i + qmax_i sig_j),
        dq_i = sum over near-tie c of q_i of step kmax_c,
        sig_j = sum over near-tie c of k_j of step, qmax_i = max_c |q8_ic|.
    To first order dLSE_i = sum_j P_ij dS_ij and dP_ij = P_ij (dS_ij -
    dLSE_i); the second order is covered by the factor exp(2 max_j |dS_ij|).
    Returns (lse_bound [B, Hq, Nq], o_bound [B, Nq, Hq, d]) of the flips,
    using the attention P of the dequantised problem (qd, kd)."""
    B, Nq, Hq, d = qn.shape
    _, Nk, Hkv, _ = kn.shape
    if not incoherent:
        return np.zeros((B, Hq, Nq)), np.zeros((B, Nq, Hq, d))
    g = Hq // Hkv
    qt, kt = f8.hadamard(qn), f8.hadamard(kn)
    sq = f8.pow2_scale(np.abs(qt).max(axis=(1, 3)))
    sk = f8.pow2_scale(np.abs(kt).max(axis=(1, 3)))
    uq, uk = qt / sq[:, None, :, None], kt / sk[:, None, :, None]
    tq, stq = near_tie(uq, 2.0 ** -21 * np.linalg.norm(uq, axis=-1, keepdims=True) + 2.0 ** -23 * np.abs(uq))
    tk, stk = near_tie(uk, 2.0 ** -21 * np.linalg.norm(uk, axis=-1, keepdims=True) + 2.0 ** -23 * np.abs(uk))
    q8, k8 = f8.e4m3(uq), f8.e4m3(uk)
    sig = (tk * stk).sum(axis=-1, keepdims=True)                       # [B, Nk, Hkv, 1]
    p_sig, _ = attn_ref.forward(qd, kd, np.broadcast_to(sig, kd.shape), scale, causal)
    p_sigv, _ = attn_ref.forward(qd, kd, sig * np.abs(vd), scale, causal)
    p_v = f8.pv_abs(qd, kd, vd, scale, causal)
    lse_b = np.zeros((B, Hq, Nq))
    o_b = np.zeros((B, Nq, Hq, d))
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            f = abs(scale) * sq[b, h] * sk[b, kv]
            kmax = np.abs(k8[b, :, kv, :]).max(axis=0)
            dq = (tq[b, :, h, :] * stq[b, :, h, :] * kmax).sum(axis=1)     # [Nq]
            qmax = np.abs(q8[b, :, h, :]).max(axis=1)                     # [Nq]
            grow = np.exp(2 * f * (dq + qmax * sig[b, :, kv, 0].max()))
            L = f * (dq + qmax * p_sig[b, :, h, 0])
            lse_b[b, h] = grow * L
            o_b[b, :, h, :] = grow[:, None] * (f * (dq[:, None] * p_v[b, :, h, :] + qmax[:, None] * p_sigv[b, :, h, :])
                                               + L[:, None] * p_v[b, :, h, :])
    return lse_b, o_b


def check_against_oracle(go, glse, x, causal, incoherent, scale, mean_check=True):
    """Bounds, with the GPU and the oracle rounding Q M, K M, V to the same
    e4m3 codes except where flip_terms allows a code to differ:
      O elementwise: |err| <= 2^-4 sum_j P_ij |V_jc| (rounding P to e4m3,
        worst case) + 2^-8 |O| (bf16 output) + 1e-4 (fp32 accumulation)
        + the flip term;
      O mean: at most twice the expected |error| of independent P rounding;
      LSE: the same -inf rows; |err| <= 1e-5 (fp32 accumulation and
        ex2.approx) + the flip term, and the mean within the mean of that."""
    qn, kn, vn = (x[n].double().numpy() for n in ("q", "k", "v"))
    ro, rlse, (qd, kd, vd) = f8.forward_fp8(qn, kn, vn, scale, causal, incoherent=incoherent)
    lse_flip, o_flip = flip_terms(qn, kn, vd, qd, kd, scale, causal, incoherent)
    bound = 2.0 ** -4 * f8.pv_abs(qd, kd, vd, scale, causal) + 2.0 ** -8 * np.abs(ro) + 1e-4 + o_flip
    err = np.abs(go - ro)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (f"worst |err| {err[worst]:.3e} > bound {bound[worst]:.3e} at {worst}; "
                                  f"max-abs {err.max():.3e}, mean-abs {err.mean():.3e}")
    if mean_check:
        expect = float(np.mean(rounding_sd(qd, kd, vd, scale, causal))) * np.sqrt(2 / np.pi)
        assert float(err.mean()) <= 2 * expect + 5e-4, (err.mean(), expect)
    fin = np.isfinite(rlse)  # rows that see no key: -inf on both sides
    assert np.array_equal(np.isfinite(glse), fin) and np.all(glse[~fin] == rlse[~fin])
    lerr = np.abs(glse - np.where(fin, rlse, 0.0))
    lb = 1e-5 + lse_flip
    assert np.all(lerr[fin] <= lb[fin]), (float(np.max(lerr[fin] - lb[fin])), float(lerr[fin].max()),
                                          float(lb[fin].max()))
    assert float(lerr[fin].mean()) <= float(lb[fin].mean()), (float(lerr[fin].mean()), float(lb[fin].mean()))


SHAPES = [
    # B, Hq, Hkv, Nq, Nk
    (1, 2, 2, 256, 256),
    (1, 4, 2, 300, 300),
    (2, 2, 1, 129, 700),
    (1, 2, 2, 700, 129),
]


@pytest.mark.parametrize("incoherent", [True, False])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fp8_matches_oracle(fa, shape, causal, incoherent):
    B, Hq, Hkv, Nq, Nk = shape
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, 128, seed=sum(shape) + 2 * causal + incoherent)
    scale = 1.0 / math.sqrt(128)
    go, glse = fp8_case(fa, x, causal, incoherent, scale)
    check_against_oracle(go, glse, x, causal, incoherent, scale)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_negative_scale(fa, causal):
    """A negative scale: S = (-Q) K^T through the instruction descriptor."""
    x = workloads.make_inputs(1, 4, 2, 300, 300, 128, seed=321 + causal)
    scale = -1.0 / math.sqrt(128)
    go, glse = fp8_case(fa, x, causal, True, scale)
    check_against_oracle(go, glse, x, causal, True, scale)


def test_fp8_full_size_sampled(fa):
    """The non-causal B=4, H=16, N=2048 workload through the FP8 path: finite
    everywhere, two heads against the oracle."""
    w = workloads.WORKLOADS[1]
    x = workloads.workload_inputs(w)
    go, glse = fp8_case(fa, x, False, True, w.scale)
    assert np.isfinite(go).all() and np.isfinite(glse).all()
    for b, h in [(0, 0), (3, 15)]:
        sl = {n: x[n][b:b + 1, :, h:h + 1] for n in ("q", "k", "v")}
        check_against_oracle(go[b:b + 1, :, h:h + 1], glse[b:b + 1, h:h + 1], sl, False, True, w.scale,
                             mean_check=False)


def test_fp8_causal_full_size_sampled(fa):
    """The causal B=2, H=16, N=8192 workload through the FP8 path: finite
    everywhere, two heads against the oracle."""
    w = workloads.WORKLOADS[2]
    x = workloads.workload_inputs(w)
    go, glse = fp8_case(fa, x, True, True, w.scale)
    assert np.isfinite(go).all() and np.isfinite(glse).all()
    for b, h in [(0, 3), (1, 12)]:
        sl = {n: x[n][b:b + 1, :, h:h + 1] for n in ("q", "k", "v")}
        check_against_oracle(go[b:b + 1, :, h:h + 1], glse[b:b + 1, h:h + 1], sl, True, True, w.scale,
                             mean_check=False)


def test_fp8_incoherent_lowers_error_with_outliers(fa):
    """Against the exact bf16-input attention: with outlier channels in Q
    and K, the incoherent transform lowers the FP8 error."""
    B, H, N, d = 1, 4, 512, 128
    x = workloads.make_inputs(B, H, H, N, N, d, seed=77)
    for n in ("q", "k"):
        t = x[n].float()
        t[..., [5, 90]] *= 20.0
        x[n] = t.to(torch.bfloat16)
    scale = 0.5 / math.sqrt(d)
    exact, _ = attn_ref.forward(*(x[n].double().numpy() for n in ("q", "k", "v")), scale, False)
    err = {}
    for inc in (False, True):
        go, _ = fp8_case(fa, x, False, inc, scale)
        err[inc] = float(np.sqrt(np.mean((go - exact) ** 2)))
    assert err[True] * 1.5 < err[False], err
