"""Plain CPU model of the FP8 (e4m3) forward with incoherent processing.

TEST INFRASTRUCTURE ONLY, like ``attn_ref``: only the test suite, the smoke
check and the benchmark's CPU leg may import it; the CUDA path shares no
code with it.

What it computes (the FlashAttention-3 summary on news.hada.io, sections
on FP8 and "incoherent processing"; the FlashAttention-4 article names the
same low-precision path): Q and K are multiplied by one random orthogonal
matrix M = diag(signs) H_d / sqrt(d) (H_d the Sylvester-Hadamard matrix) so
that outlier channels are spread before quantisation; since M M^T = I,
(Q M)(K M)^T = Q K^T and the attention is unchanged in exact arithmetic.
Q M, K M and V are then scaled per (batch, head) by the smallest power of
two that brings their largest magnitude to at most 448 (the largest finite
e4m3 value), i.e. into (224, 448], and rounded to e4m3 (round to nearest,
ties to even, saturating). The attention of the
dequantised tensors (values times their scales) is the reference this
module returns; the GPU path additionally rounds P to e4m3 for the P V
GEMM, an error the tests bound separately (``pv_abs``).

Readings where the pages are silent:
  * one scale per (batch, head) and tensor, a power of two: dividing by it
    is exact, so a code is the round-to-nearest-even of x / s whatever
    precision the division is done in (a scale of amax / 448 would let the
    rounding of the division decide ties, which bf16 inputs hit often);
  * the signs: sign_i = -1 where bit 31 of (2654435769 * (i + 1)) mod 2^32
    is set, else +1 (a fixed counter-based sequence, the same on both
    sides);
  * the transform is applied along the head dimension d (a power of two).
"""
from __future__ import annotations

import numpy as np
import scipy.linalg

from oracle import attn_ref

__all__ = ["E4M3_MAX", "hadamard_signs", "hadamard", "e4m3", "pow2_scale", "quantize_per_head", "forward_fp8",
           "pv_abs"]

E4M3_MAX = 448.0


def hadamard_signs(d: int) -> np.ndarray:
    i = np.arange(d, dtype=np.uint64)
    h = (np.uint64(2654435769) * (i + np.uint64(1))) & np.uint64(0xFFFFFFFF)
    return np.where((h >> np.uint64(31)) & np.uint64(1), -1.0, 1.0)


def hadamard(x: np.ndarray) -> np.ndarray:
    """x @ diag(signs) H_d / sqrt(d) along the last axis (fp64)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    M = hadamard_signs(d)[:, None] * scipy.linalg.hadamard(d).astype(np.float64) / np.sqrt(d)
    return x @ M


def e4m3(x: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even), saturating at +-448.
    e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; normal
    values 2^(e-7) (1 + m/8) for e = 1..15 (448 = 2^8 * 1.75 the largest
    finite), subnormals 2^-6 * m/8."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)           # below 2^-6 the step stays 2^-9 (subnormals)
    step = np.exp2(e - 3.0)           # 3 mantissa bits
    q = np.round(a / step) * step     # numpy rounds half to even
    q = np.minimum(q, E4M3_MAX)
    return np.where(x < 0, -q, q)


def pow2_scale(amax: np.ndarray) -> np.ndarray:
    """The smallest power of two s with amax / s <= 448 (1 where amax = 0):
    s = 2^ceil(log2(amax / 448)), computed exactly from amax = m 2^E with m
    in [1/2, 1) and 448 = (7/8) 2^9: s = 2^(E - 9) if m <= 7/8 else 2^(E - 8)."""
    amax = np.asarray(amax, dtype=np.float64)
    m, E = np.frexp(amax)
    e = np.where(m <= 0.875, E - 9, E - 8)
    return np.where(amax > 0, np.ldexp(1.0, e), 1.0)


def quantize_per_head(x: np.ndarray):
    """x [B, N, H, d] -> (e4m3 values as fp64, scales [B, H]): each head's
    scale is pow2_scale(amax(|x[b, :, h, :]|)), so its largest magnitude maps
    into (224, 448] (scale 1 for an all-zero head)."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.abs(x).max(axis=(1, 3))                      # [B, H]
    s = pow2_scale(amax)
    q = e4m3(x / s[:, None, :, None])
    return q, s


def forward_fp8(q, k, v, scale: float, causal: bool, incoherent: bool = True):
    """O and LSE of the attention of the dequantised e4m3 tensors, plus the
    dequantised tensors (qd, kd, vd) for bounding the GPU's P rounding."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if incoherent:
        q, k = hadamard(q), hadamard(k)
    q8, sq = quantize_per_head(q)
    k8, sk = quantize_per_head(k)
    v8, sv = quantize_per_head(v)
    qd = q8 * sq[:, None, :, None]
    kd = k8 * sk[:, None, :, None]
    vd = v8 * sv[:, None, :, None]
    o, lse = attn_ref.forward(qd, kd, vd, scale, causal)
    return o, lse, (qd, kd, vd)


def pv_abs(qd, kd, vd, scale: float, causal: bool) -> np.ndarray:
    """sum_j P_ij |V_j| per output element ([B, Nq, Hq, d]): rounding each P
    to e4m3 moves O_i by at most 2^-4 of this (3 mantissa bits)."""
    o, _ = attn_ref.forward(qd, kd, np.abs(vd), scale, causal)
    return o
