"""Helpers shared by the GPU parity tests (comparison and tolerances)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances for bf16 I/O with fp32 accumulation: max-abs 2e-2 and mean-abs
# 2e-3 on O, dQ, dK, dV; 1e-3 absolute on LSE (natural log).
TOL_MAX = 2e-2
TOL_MEAN = 2e-3
TOL_LSE = 1e-3


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def rounding_floor(ref: np.ndarray) -> float:
    """max |bf16(ref) - ref|: the part of the error output rounding alone causes."""
    r = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    return float(np.abs(r - ref).max()) if ref.size else 0.0


def assert_close(name: str, got: np.ndarray, ref: np.ndarray, max_tol=TOL_MAX, mean_tol=TOL_MEAN):
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if ref.size == 0:
        return
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{name}: non-finite pattern differs"
    diff = np.abs(got[fin] - ref[fin])
    mx, mean = float(diff.max()) if diff.size else 0.0, float(diff.mean()) if diff.size else 0.0
    assert mx <= max_tol and mean <= mean_tol, (
        f"{name}: max-abs {mx:.3e} (tol {max_tol}), mean-abs {mean:.3e} (tol {mean_tol}), "
        f"bf16 rounding floor {rounding_floor(ref[fin]):.3e}")
    if not fin.all():
        assert np.array_equal(got[~fin], ref[~fin]), f"{name}: infinite entries differ"


def assert_lse(got: np.ndarray, ref: np.ndarray, tol=TOL_LSE):
    assert_close("lse", got, ref, max_tol=tol, mean_tol=tol)


def assert_close_scaled(name: str, got: np.ndarray, ref: np.ndarray, max_tol=TOL_MAX, mean_tol=TOL_MEAN,
                        rel=2.0 ** -8, extra=0.0):
    """For outputs that grow past |x| = 4, where bf16's ulp (2^-7 |x| at
    most) makes the fixed max-abs bound smaller than output rounding allows
    (long causal GQA backward: dV and dK of the first keys sum over every
    query of the group; Q, K with σ = 2: nearly one-hot rows and large dQ):
    each element within max_tol + rel * |ref| (rel = 2^-8 by default, i.e.
    between half an ulp and one ulp of the reference value) + `extra` (an
    elementwise allowance derived by the caller), mean-abs within mean_tol as
    for the workloads. The failure message reports the bf16
    rounding floor and how many elements exceed the fixed max_tol."""
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all() and np.isfinite(ref).all(), name
    diff = np.abs(got - ref)
    bound = max_tol + np.abs(ref) * rel + extra
    worst = int(np.argmax(diff - bound))
    mean = float(diff.mean())
    assert (diff <= bound).all() and mean <= mean_tol, (
        f"{name}: worst element |err| {diff.flat[worst]:.3e} at |ref| {abs(ref.flat[worst]):.3e} "
        f"(bound {bound.flat[worst]:.3e}), max-abs {float(diff.max()):.3e}, mean-abs {mean:.3e} (tol {mean_tol}), "
        f"bf16 rounding floor {rounding_floor(ref):.3e}, {int((diff > max_tol).sum())} elements above {max_tol}")


def error_report(got: np.ndarray, ref: np.ndarray, max_tol=TOL_MAX) -> dict:
    """max-abs and mean-abs error, the bf16 rounding floor of the reference,
    its largest magnitude, and how many elements exceed max_tol."""
    diff = np.abs(got - ref)
    return {"max_abs": float(diff.max()), "mean_abs": float(diff.mean()), "floor": rounding_floor(ref),
            "max_ref": float(np.abs(ref).max()), "n_above_tol": int((diff > max_tol).sum()), "n": int(diff.size)}



def d_term_bounds(q, k, do, o_gpu, o_exact, scale, causal):
    """Gradient error that comes from D_i = sum_c dO_ic O_ic being formed
    from the bf16 O the backward receives (the oracle forms it from its own
    fp64 O). With dD_i = sum_c dO_ic (O_gpu - O_exact)_ic every dS_ij moves by
    -P_ij dD_i, so
        |d dQ_ic| <= scale |dD_i| sum_j P_ij |K_jc|
        |d dK_jc| <= scale sum_(i, h in the group) P_ij |dD_i| |Q_ic|
    (dV does not involve D). Arrays are fp64 BSHD of one kv group: q, do,
    o_gpu, o_exact [B, N, G, d], k [B, N, 1, d]. Both sums are attention
    products the oracle already computes: P |K| is the forward with V = |K|,
    sum_i P_ij X_i is the dV of the backward with dO = X."""
    from oracle import attn_ref
    dD = np.abs(np.sum(do * (o_gpu - o_exact), axis=-1, keepdims=True))
    p_absk, _ = attn_ref.forward(q, k, np.abs(k), scale, causal)
    bdq = scale * dD * p_absk
    _, _, pt_x = attn_ref.backward(q, k, k, dD * np.abs(q), scale, causal)
    bdk = scale * pt_x
    return bdq, bdk
