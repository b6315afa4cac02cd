"""Pins of the FP8 oracle (oracle/attn_fp8_ref.py) to things fixed outside
it: torch's e4m3 conversion, the saturation rule, the orthogonality of the
incoherent transform and the exactness it implies, and the error reduction
it is meant to bring on inputs with outlier channels (CPU only)."""
import numpy as np
import pytest
import torch

from oracle import attn_fp8_ref as f8
from oracle import attn_ref


def test_e4m3_matches_torch_conversion():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 30, 4000), rng.normal(0, 0.01, 2000), rng.uniform(-448, 448, 2000),
                        np.array([0.0, 1.0625, 1.03125, 1.09375, 2.0 ** -10, 3 * 2.0 ** -10, 448.0, -448.0])])
    x = x[np.abs(x) <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(f8.e4m3(x), want)


def test_e4m3_saturates():
    np.testing.assert_array_equal(f8.e4m3(np.array([1000.0, -460.0, 449.0, 1e30])), [448.0, -448.0, 448.0, 448.0])


def test_hadamard_signs_first_values():
    # bit 31 of 2654435769 * (i + 1) mod 2^32, computed with Python integers
    want = [-1.0 if ((2654435769 * (i + 1)) % 2 ** 32) >> 31 else 1.0 for i in range(128)]
    np.testing.assert_array_equal(f8.hadamard_signs(128), want)
    assert 40 < int((f8.hadamard_signs(128) < 0).sum()) < 88  # a mix of both signs


def test_hadamard_is_orthogonal_and_keeps_scores():
    d = 128
    M = f8.hadamard(np.eye(d))
    np.testing.assert_allclose(M @ M.T, np.eye(d), atol=1e-12)
    # row i of the transform is sign_i * H[i, :] / sqrt(d), H[0, :] all ones
    np.testing.assert_allclose(M[0], f8.hadamard_signs(d)[0] * np.ones(d) / np.sqrt(d), atol=1e-15)
    rng = np.random.default_rng(2)
    q, k = rng.normal(size=(5, d)), rng.normal(size=(7, d))
    np.testing.assert_allclose(f8.hadamard(q) @ f8.hadamard(k).T, q @ k.T, atol=1e-11)


def test_incoherent_transform_leaves_attention_unchanged():
    rng = np.random.default_rng(3)
    q, k, v = (rng.normal(size=(1, 40, 2, 128)) for _ in range(3))
    for causal in (False, True):
        o1, l1 = attn_ref.forward(q, k, v, 0.09, causal)
        o2, l2 = attn_ref.forward(f8.hadamard(q), f8.hadamard(k), v, 0.09, causal)
        np.testing.assert_allclose(o2, o1, atol=1e-12)
        np.testing.assert_allclose(l2, l1, atol=1e-12)


def test_pow2_scale_is_the_smallest_power_of_two():
    """Checked with exact rational arithmetic: s is a power of two, amax / s
    <= 448, and amax / (s / 2) > 448."""
    from fractions import Fraction
    rng = np.random.default_rng(9)
    vals = np.concatenate([rng.uniform(1e-3, 1e3, 500), [448.0, 224.0, 224.00000000001, 5.25, 4.53125, 1.0, 2.0 ** -20,
                                                         448.0 * 2 ** 7, 447.9999, 392.0, 392.5]])
    for a, s in zip(vals, f8.pow2_scale(vals)):
        fs = Fraction(float(s))
        assert fs.numerator == 1 or fs.denominator == 1, s
        assert (fs.numerator & (fs.numerator - 1)) == 0 and (fs.denominator & (fs.denominator - 1)) == 0, s
        assert Fraction(float(a)) / fs <= 448 < Fraction(float(a)) / (fs / 2), (a, s)
    assert f8.pow2_scale(np.array([0.0]))[0] == 1.0


def test_quantize_per_head():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(2, 50, 3, 128)) * np.array([1.0, 10.0, 0.01])[None, None, :, None]
    q, s = f8.quantize_per_head(x)
    top = np.abs(q).max(axis=(1, 3))
    assert np.all((top > 224.0) & (top <= 448.0))                     # each head's amax maps into (224, 448]
    np.testing.assert_array_equal(f8.e4m3(q), q)                       # already e4m3 values
    np.testing.assert_array_equal(q, f8.e4m3(x / s[:, None, :, None]))  # exact division by a power of two
    deq = q * s[:, None, :, None]
    big = np.abs(x) > 2.0 ** -6 * s[:, None, :, None]                  # normal range: half an ulp relative
    assert np.all(np.abs(deq - x)[big] <= 2.0 ** -4 * np.abs(x)[big] + 1e-15)
    z, sz = f8.quantize_per_head(np.zeros((1, 4, 1, 8)))
    assert np.all(z == 0) and np.all(sz == 1.0)


def test_codes_of_bf16_inputs_do_not_depend_on_the_division_precision():
    """With a power-of-two scale, x / s in fp32 (as a GPU computes it) and in
    fp64 give the same e4m3 code for every bf16 x, including the exact ties
    that bf16 values hit (e.g. amax = 5.25, where amax / 448 is 3/256)."""
    rng = np.random.default_rng(10)
    x = torch.from_numpy(rng.normal(size=(1, 700, 1, 128))).to(torch.bfloat16).double().numpy()
    x[0, 0, 0, 0] = 5.25
    q64, s = f8.quantize_per_head(x)
    x32 = torch.from_numpy(x).float() / torch.from_numpy(s).float()[:, None, :, None]
    q32 = x32.to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(q32, q64)


def test_incoherent_processing_lowers_fp8_error_with_outliers():
    """The point of the transform: with a few outlier channels in Q and K,
    the FP8 attention error against the exact result drops."""
    rng = np.random.default_rng(5)
    B, N, H, d = 1, 256, 2, 128
    q, k, v = (rng.normal(size=(B, N, H, d)) for _ in range(3))
    for t in (q, k):
        t[..., [3, 77]] *= 30.0
    scale = 0.5 / np.sqrt(d)
    exact, _ = attn_ref.forward(q, k, v, scale, False)
    err = {}
    for inc in (False, True):
        o, _, _ = f8.forward_fp8(q, k, v, scale, False, incoherent=inc)
        err[inc] = float(np.sqrt(np.mean((o - exact) ** 2)))
    assert err[True] * 1.5 < err[False], err


@pytest.mark.parametrize("causal", [False, True])
def test_pv_abs_bounds_p_rounding(causal):
    """Rounding every P to e4m3 moves O by at most 2^-4 sum_j P_ij |V_j|."""
    rng = np.random.default_rng(6)
    q, k, v = (rng.normal(size=(1, 30, 1, 16)) for _ in range(3))
    scale = 0.25
    P = attn_ref.probabilities(q[0, :, 0], k[0, :, 0], scale, causal)
    o_exact = P @ v[0, :, 0]
    o_p8 = f8.e4m3(P * 256.0) / 256.0 @ v[0, :, 0]  # P scaled into the normal e4m3 range, as the kernel's 2^(x-m)
    bound = f8.pv_abs(q, k, v, scale, causal)[0, :, 0]
    assert np.all(np.abs(o_p8 - o_exact) <= 2.0 ** -4 * bound + 1e-12)


@pytest.mark.parametrize("incoherent", [False, True])
def test_forward_fp8_scale_equivariance(incoherent):
    """forward_fp8 applies each per-head scale exactly once: multiplying Q
    (or K) of one head by a power of two leaves its e4m3 codes unchanged and
    multiplies that head's scale by the same power, so the result equals the
    call with the softmax scale multiplied instead; multiplying V by a power
    of two multiplies O by it and leaves LSE unchanged. A dropped, doubled or
    misplaced scale factor (sq, sk or sv) breaks one of these equalities."""
    rng = np.random.default_rng(7)
    B, N, H, d = 1, 48, 2, 128
    q, k, v = (rng.normal(size=(B, N, H, d)) for _ in range(3))
    scale = 0.09
    for causal in (False, True):
        o, lse, _ = f8.forward_fp8(q, k, v, scale, causal, incoherent=incoherent)
        o2, lse2, _ = f8.forward_fp8(4.0 * q, k, v, scale, causal, incoherent=incoherent)
        o3, lse3, _ = f8.forward_fp8(q, k, v, 4.0 * scale, causal, incoherent=incoherent)
        np.testing.assert_allclose(o2, o3, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse2, lse3, rtol=0, atol=1e-12)
        o4, lse4, _ = f8.forward_fp8(q, 0.5 * k, v, scale, causal, incoherent=incoherent)
        o5, lse5, _ = f8.forward_fp8(q, k, v, 0.5 * scale, causal, incoherent=incoherent)
        np.testing.assert_allclose(o4, o5, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse4, lse5, rtol=0, atol=1e-12)
        o6, lse6, _ = f8.forward_fp8(q, k, 8.0 * v, scale, causal, incoherent=incoherent)
        np.testing.assert_allclose(o6, 8.0 * o, rtol=0, atol=1e-11)
        np.testing.assert_allclose(lse6, lse, rtol=0, atol=0)
        assert not np.allclose(o2, o, atol=1e-3)  # the factor does reach the logits


@pytest.mark.parametrize("incoherent", [False, True])
def test_forward_fp8_close_to_exact_attention(incoherent):
    """On ordinary N(0, 1) inputs the FP8 result stays within the e4m3
    quantisation error of the exact attention. First-order estimate: every
    element of Q M, K M and V carries a relative rounding error of rms at
    most 2^-4 / sqrt(3) (uniform within half an ulp of a 3-bit mantissa), so
    a logit s = scale * q.k moves by about scale * sqrt(2 d) * 2^-4 / sqrt(3)
    (about 0.05 here) and O by that much of the spread of V under P (below
    1) plus V's own 2^-4 / sqrt(3) relative error averaged over the attended
    keys: a relative rms error of O of a few percent, far below the 100 % of
    a lost scale factor and above zero (quantisation did happen)."""
    rng = np.random.default_rng(8)
    B, N, H, d = 1, 256, 2, 128
    q, k, v = (rng.normal(size=(B, N, H, d)) for _ in range(3))
    scale = 1.0 / np.sqrt(d)
    for causal in (False, True):
        exact, lse_exact = attn_ref.forward(q, k, v, scale, causal)
        o, lse, _ = f8.forward_fp8(q, k, v, scale, causal, incoherent=incoherent)
        est = scale * np.sqrt(2 * d) * 2.0 ** -4 / np.sqrt(3)
        rel = float(np.sqrt(np.mean((o - exact) ** 2)) / np.sqrt(np.mean(exact ** 2)))
        assert 1e-3 < rel < 2 * (est + 2.0 ** -4 / np.sqrt(3)), (causal, rel, est)
        assert float(np.abs(lse - lse_exact).max()) < 8 * est, (causal, float(np.abs(lse - lse_exact).max()))


@pytest.mark.parametrize("which", [0, 1, 2])
def test_planted_dropped_scale_fails_a_pin(monkeypatch, which):
    """A planted mistake: forward_fp8 dequantising one of Q, K, V without its
    per-head scale (the codes themselves are right). The equivariance or the
    closeness pin must fail."""
    real = f8.quantize_per_head
    calls = {"n": 0}

    def broken(x):
        codes, s = real(x)
        i = calls["n"] % 3
        calls["n"] += 1
        return (codes, np.ones_like(s)) if i == which else (codes, s)

    monkeypatch.setattr(f8, "quantize_per_head", broken)
    failed = 0
    for pin in (test_forward_fp8_scale_equivariance, test_forward_fp8_close_to_exact_attention):
        try:
            calls["n"] = 0
            pin(True)
        except AssertionError:
            failed += 1
    assert failed >= 1
