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


def test_quantize_per_head():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(2, 50, 3, 128)) * np.array([1.0, 10.0, 0.01])[None, None, :, None]
    q, s = f8.quantize_per_head(x)
    np.testing.assert_array_equal(np.abs(q).max(axis=(1, 3)), 448.0)  # each head's amax maps to 448
    np.testing.assert_array_equal(f8.e4m3(q), q)                       # already e4m3 values
    deq = q * s[:, None, :, None]
    big = np.abs(x) > 2.0 ** -6 * s[:, None, :, None]                  # normal range: half an ulp relative
    assert np.all(np.abs(deq - x)[big] <= 2.0 ** -4 * np.abs(x)[big] + 1e-15)
    z, sz = f8.quantize_per_head(np.zeros((1, 4, 1, 8)))
    assert np.all(z == 0) and np.all(sz == 1.0)


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
