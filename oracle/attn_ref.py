"""Plain fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check of the
package entry point, and the CPU-baseline leg of the benchmark may import
this module. The CUDA path never calls it and shares no code with it.

What it computes (the plain definition, written out):
  The post "FlashAttention v1" (deep_school, post #630), section
  "Проблема базового attention", names scaled dot-product attention and
  says the standard implementation builds the full n x n matrix QK^T; its
  formula image was not preserved, so the textbook definition is used:

      S   = scale * Q K^T                       (materialised, fp64)
      S_ij = -inf where key j is hidden by the causal mask
      m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i)
      P   = exp(S - m) / l                      (row softmax)
      O   = P V,          LSE_i = m_i + ln l_i  (natural log)

  The same post, sections "Идея FlashAttention" and "Онлайн-Softmax", states
  that the tiled method with online softmax gives a result fully equal to
  this classical softmax, so the oracle is the definition itself, not the
  tiled algorithm. ``blockwise_forward`` below restates the online-softmax
  update (running max, running sum, rescale of the accumulated output when
  the max grows) only to check that claim.

  Backward (the FlashAttention-3 summary on news.hada.io, section "Resumo do
  FlashAttention": tiling plus recomputation) reaches the analytic gradients
  of the same function:

      dV_g = sum_{h in group g} P_h^T dO_h
      dP   = dO_h V_g^T
      D_i  = sum_c dO_ic O_ic
      dS   = P o (dP - D)
      dQ_h = scale * dS K_g
      dK_g = scale * sum_{h in group g} dS_h^T Q_h

Readings where the pages are silent:
  * causal alignment is bottom-right: key j is visible to query i iff
    j <= i + (Nk - Nq); with Nq == Nk this is j <= i;
  * sliding windows (local attention; the FlashAttention-4 article and the
    FA-2 notes name variable and sliding-window masks without defining
    them): with the same bottom-right offset, key j is visible to query i
    iff i + off - window_left <= j <= i + off + window_right, off = Nk - Nq,
    a negative bound meaning no limit on that side; causal is
    window_right = 0 with no left limit;
  * grouped-query attention maps query head h to kv head h // (Hq // Hkv);
  * a row with no visible key has O = 0 and LSE = -inf and contributes no
    gradient.

Arrays are numpy, BSHD layout: q, o, dO [B, Nq, Hq, d]; k, v [B, Nk, Hkv, d];
lse [B, Hq, Nq]. Everything is computed in float64.
"""
from __future__ import annotations

import numpy as np

__all__ = ["visible_mask", "probabilities", "forward", "backward", "backward_abs_terms", "blockwise_forward"]

PANEL_ROWS = 1024  # rows of S formed at a time (memory bound only; every entry is formed)


def _group(hq: int, hkv: int) -> int:
    if hkv <= 0 or hq % hkv != 0:
        raise ValueError(f"Hq={hq} must be a positive multiple of Hkv={hkv}")
    return hq // hkv


def _window(causal: bool, window):
    """(left, right) bounds, negative = unbounded; causal forces right = 0."""
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    if causal:
        wr = 0 if wr < 0 else min(wr, 0)
    return wl, wr


def visible_mask(rows: np.ndarray, nq: int, nk: int, causal: bool, window=None) -> np.ndarray:
    """Boolean [len(rows), nk]: True where key j is visible to query row i.
    ``window`` = (left, right) as in the module notes (None: no window)."""
    rows = np.asarray(rows, dtype=np.int64)
    wl, wr = _window(causal, window)
    j = np.arange(nk, dtype=np.int64)[None, :]
    diag = rows[:, None] + (nk - nq)
    vis = np.ones((rows.shape[0], nk), dtype=bool)
    if wr >= 0:
        vis &= j <= diag + wr
    if wl >= 0:
        vis &= j >= diag - wl
    return vis


def _scores(Q: np.ndarray, K: np.ndarray, scale: float, rows: np.ndarray, nq: int, causal: bool,
            window=None) -> np.ndarray:
    S = scale * (Q @ K.T)
    wl, wr = _window(causal, window)
    if wl >= 0 or wr >= 0:
        S = np.where(visible_mask(rows, nq, K.shape[0], causal, window), S, -np.inf)
    return S


def _softmax_stats(S: np.ndarray):
    """Row max m, row sum l of exp(S - m), and P; empty rows give P = 0."""
    m = S.max(axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    E = np.exp(S - m_safe[:, None])  # exp(-inf) = 0 for masked entries
    l = E.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        P = np.where(finite[:, None], E / np.where(l > 0, l, 1.0)[:, None], 0.0)
        lse = np.where(finite, m_safe + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return P, lse


def _softmax_grad(P: np.ndarray, dP: np.ndarray, D: np.ndarray) -> np.ndarray:
    """dS = P o (dP - D), with D_i = sum_j P_ij dP_ij = sum_c dO_ic O_ic."""
    return P * (dP - D[:, None])


def probabilities(Q: np.ndarray, K: np.ndarray, scale: float, causal: bool, window=None) -> np.ndarray:
    """P for one head: Q [Nq, d], K [Nk, d] -> [Nq, Nk] (fp64)."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    nq = Q.shape[0]
    S = _scores(Q, K, scale, np.arange(nq), nq, causal, window)
    P, _ = _softmax_stats(S)
    return P


def forward(q, k, v, scale: float, causal: bool, rows=None, window=None):
    """O and LSE. ``rows`` optionally restricts the query rows computed
    (indices into Nq); the outputs then have len(rows) in place of Nq.
    ``window`` = (left, right) sliding-window bounds (module notes)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, dk = k.shape
    assert dk == d and v.shape == k.shape
    g = _group(Hq, Hkv)
    rows = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    R = rows.shape[0]
    o = np.zeros((B, R, Hq, d))
    lse = np.empty((B, Hq, R))
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            K = k[b, :, kv, :]
            V = v[b, :, kv, :]
            for r0 in range(0, R, PANEL_ROWS):
                rr = rows[r0:r0 + PANEL_ROWS]
                S = _scores(q[b, rr, h, :], K, scale, rr, Nq, causal, window)
                P, l = _softmax_stats(S)
                o[b, r0:r0 + len(rr), h, :] = P @ V
                lse[b, h, r0:r0 + len(rr)] = l
    return o, lse


def backward(q, k, v, do, scale: float, causal: bool, window=None):
    """Analytic dQ, dK, dV of L = sum(dO * O) (fp64, oracle's own O)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    g = _group(Hq, Hkv)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rows_all = np.arange(Nq)
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            K = k[b, :, kv, :]
            V = v[b, :, kv, :]
            for r0 in range(0, Nq, PANEL_ROWS):
                rr = rows_all[r0:r0 + PANEL_ROWS]
                Q = q[b, rr, h, :]
                dO = do[b, rr, h, :]
                S = _scores(Q, K, scale, rr, Nq, causal, window)
                P, _ = _softmax_stats(S)
                O = P @ V
                D = np.sum(dO * O, axis=1)
                dP = dO @ V.T
                dS = _softmax_grad(P, dP, D)
                dv[b, :, kv, :] += P.T @ dO
                dq[b, rr, h, :] = scale * (dS @ K)
                dk[b, :, kv, :] += scale * (dS.T @ Q)
    return dq, dk, dv


def backward_abs_terms(q, k, v, do, scale: float, causal: bool, window=None):
    """Magnitudes that bound how much rounding the intermediates P and dS
    (relative error at most e per element) can move the gradients, per
    output element, formed from the same quantities as ``backward``:

        a_dq[b, i, h, c] = scale * sum_j |dS_ij| |K_jc|
        a_dk[b, j, g, c] = scale * sum_{h in g} sum_i |dS_ij| |Q_ic|
        a_dv[b, j, g, c] = sum_{h in g} sum_i P_ij |dO_ic|

    (triangle inequality on dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO:
    rounding every dS_ij to dS_ij (1 + e_ij) with |e_ij| <= e moves dQ_ic by
    at most e a_dq[i, c]; likewise dK, and dV for P). Test infrastructure
    for the error bounds of the GPU comparisons."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    g = _group(Hq, Hkv)
    a_dq = np.zeros_like(q)
    a_dk = np.zeros_like(k)
    a_dv = np.zeros_like(v)
    rows_all = np.arange(Nq)
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            K = k[b, :, kv, :]
            V = v[b, :, kv, :]
            for r0 in range(0, Nq, PANEL_ROWS):
                rr = rows_all[r0:r0 + PANEL_ROWS]
                Q = q[b, rr, h, :]
                dO = do[b, rr, h, :]
                S = _scores(Q, K, scale, rr, Nq, causal, window)
                P, _ = _softmax_stats(S)
                O = P @ V
                D = np.sum(dO * O, axis=1)
                dS = np.abs(_softmax_grad(P, dO @ V.T, D))
                a_dv[b, :, kv, :] += P.T @ np.abs(dO)
                a_dq[b, rr, h, :] = scale * (dS @ np.abs(K))
                a_dk[b, :, kv, :] += scale * (dS.T @ np.abs(Q))
    return a_dq, a_dk, a_dv


def blockwise_forward(q, k, v, scale: float, causal: bool, key_blocks):
    """Online-softmax restatement over an arbitrary partition of the keys.

    ``key_blocks`` is a list of (start, stop) covering 0..Nk in order. For
    each new block the running row max, the running sum of exponentials and
    the accumulated output are updated; the accumulated output is rescaled
    by exp(m_old - m_new) when the block raises the max (the three bullets
    of section "Онлайн-Softmax" of the FlashAttention v1 post)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    g = _group(Hq, Hkv)
    o = np.zeros((B, Nq, Hq, d))
    lse = np.empty((B, Hq, Nq))
    rows = np.arange(Nq)
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            m = np.full(Nq, -np.inf)
            l = np.zeros(Nq)
            acc = np.zeros((Nq, d))
            for (s0, s1) in key_blocks:
                Kb = k[b, s0:s1, kv, :]
                Vb = v[b, s0:s1, kv, :]
                S = scale * (q[b, :, h, :] @ Kb.T)
                if causal:
                    j = np.arange(s0, s1)[None, :]
                    S = np.where(j <= rows[:, None] + (Nk - Nq), S, -np.inf)
                m_new = np.maximum(m, S.max(axis=1))
                m_use = np.where(np.isfinite(m_new), m_new, 0.0)
                alpha = np.where(np.isfinite(m), np.exp(m - m_use), 0.0)
                Pb = np.exp(S - m_use[:, None])
                l = l * alpha + Pb.sum(axis=1)
                acc = acc * alpha[:, None] + Pb @ Vb
                m = m_new
            with np.errstate(divide="ignore", invalid="ignore"):
                o[b, :, h, :] = np.where(l[:, None] > 0, acc / np.where(l > 0, l, 1.0)[:, None], 0.0)
                lse[b, h, :] = np.where(l > 0, np.where(np.isfinite(m), m, 0.0) + np.log(np.where(l > 0, l, 1.0)),
                                        -np.inf)
    return o, lse
