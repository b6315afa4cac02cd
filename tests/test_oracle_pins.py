"""Pins for the fp64 oracle: each check ties it to something other than
itself (closed forms, invariants, hand-worked cases, brute force, finite
differences, a library routine), so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them.
The last section plants such mistakes in the oracle and checks that they are
caught."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attn_ref

HERE = os.path.dirname(os.path.abspath(__file__))
RNG = np.random.default_rng(20261202)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def tiny_problem(B=1, Hq=2, Hkv=1, Nq=5, Nk=5, d=3, s=1.0):
    return rand(B, Nq, Hq, d, scale=s), rand(B, Nk, Hkv, d, scale=s), rand(B, Nk, Hkv, d)


# ---------------------------------------------------------------- forward --

def check_worked_examples(fwd):
    with open(os.path.join(HERE, "golden", "worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = np.array(c["q"], dtype=np.float64)[None, :, None, :]
        k = np.array(c["k"], dtype=np.float64)[None, :, None, :]
        v = np.array(c["v"], dtype=np.float64)[None, :, None, :]
        o, lse = fwd(q, k, v, c["scale"], c["causal"])
        want_lse = np.array([-np.inf if x == "-inf" else x for x in c["lse"]], dtype=np.float64)
        np.testing.assert_allclose(o[0, :, 0, :], np.array(c["o"]), rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(lse[0, 0], want_lse, rtol=0, atol=1e-12, err_msg=c["name"])


def check_rows_sum_to_one(_fwd=None):
    for causal, (nq, nk) in itertools.product([False, True], [(7, 7), (4, 9), (9, 9)]):
        Q, K = rand(nq, 4, scale=3.0), rand(nk, 4, scale=3.0)
        P = attn_ref.probabilities(Q, K, 0.5, causal)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        assert (P >= 0).all()


def check_constant_v(fwd):
    for causal in (False, True):
        q, k, _ = tiny_problem(B=2, Hq=4, Hkv=2, Nq=9, Nk=9, d=5, s=2.0)
        v0 = rand(5)
        v = np.broadcast_to(v0, k.shape).copy()
        o, _ = fwd(q, k, v, 0.7, causal)
        np.testing.assert_allclose(o, np.broadcast_to(v0, o.shape), rtol=0, atol=1e-12)


def check_zero_q(fwd):
    # Q = 0: every visible logit is 0, so O_i = mean of visible V rows and LSE_i = ln(count).
    for causal, (nq, nk) in itertools.product([False, True], [(6, 6), (3, 8)]):
        B, Hq, Hkv, d = 2, 4, 2, 3
        q = np.zeros((B, nq, Hq, d))
        k, v = rand(B, nk, Hkv, d), rand(B, nk, Hkv, d)
        o, lse = fwd(q, k, v, 0.9, causal)
        for b, h, i in itertools.product(range(B), range(Hq), range(nq)):
            n_vis = (i + (nk - nq) + 1) if causal else nk
            n_vis = min(n_vis, nk)
            kv = h // (Hq // Hkv)
            np.testing.assert_allclose(o[b, i, h], v[b, :n_vis, kv].mean(axis=0), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, h, i], math.log(n_vis), rtol=0, atol=1e-12)


def check_one_hot(fwd):
    # one key with a logit far above the rest: O is that key's value row
    nk, d = 11, 4
    k = np.zeros((1, nk, 1, d))
    k[0, 6, 0, 0] = 1.0
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 80.0
    v = rand(1, nk, 1, d)
    o, lse = fwd(q, k, v, 1.0, False)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 6, 0], rtol=0, atol=1e-20 + 1e-30)
    np.testing.assert_allclose(lse[0, 0, 0], 80.0, rtol=0, atol=1e-12)


def check_causal_row0(fwd):
    q, k, v = tiny_problem(Nq=8, Nk=8, s=2.0)
    o, lse = fwd(q, k, v, 0.6, True)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0, 0], 0.6 * q[0, 0, 0] @ k[0, 0, 0], rtol=0, atol=1e-12)


def brute_force(q, k, v, scale, causal, window=None):
    """Scalar loops with math.exp and math.fsum (tiny inputs only). A row
    with no visible key gets O = 0 and LSE = -inf."""
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    g = Hq // Hkv
    o = np.zeros((B, Nq, Hq, d))
    lse = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            for i in range(Nq):
                keys = [j for j in range(Nk) if seen(i, j, Nq, Nk, causal, window)]
                if not keys:
                    lse[b, h, i] = -math.inf
                    continue
                logits = [scale * math.fsum(q[b, i, h, c] * k[b, j, h // g, c] for c in range(d)) for j in keys]
                top = max(logits)
                w = [math.exp(s - top) for s in logits]
                tot = math.fsum(w)
                lse[b, h, i] = top + math.log(tot)
                for c in range(d):
                    o[b, i, h, c] = math.fsum(w[t] * v[b, j, h // g, c] for t, j in enumerate(keys)) / tot
    return o, lse


def seen(i, j, nq, nk, causal, window):
    """Whether query i sees key j: causal keeps j <= i + nk - nq; a window
    (left, right) keeps i + nk - nq - left <= j <= i + nk - nq + right,
    a negative bound meaning no limit on that side."""
    diag = i + nk - nq
    if causal and j > diag:
        return False
    if window is not None:
        left, right = window
        if left >= 0 and j < diag - left:
            return False
        if right >= 0 and j > diag + right:
            return False
    return True


def check_brute_force(fwd):
    for causal, (nq, nk) in itertools.product([False, True], [(7, 7), (5, 12), (16, 16)]):
        q, k, v = tiny_problem(B=1, Hq=4, Hkv=2, Nq=nq, Nk=nk, d=3, s=1.5)
        o, lse = fwd(q, k, v, 0.8, causal)
        o_bf, lse_bf = brute_force(q, k, v, 0.8, causal)
        np.testing.assert_allclose(o, o_bf, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lse_bf, rtol=0, atol=1e-12)


def torch_sdpa(q, k, v, scale, causal):
    """torch CPU fp64 scaled_dot_product_attention (math backend), BSHD in/out.
    Grouped heads are replicated; the causal mask is built bottom-right here."""
    from torch.nn.attention import SDPBackend, sdpa_kernel
    tq = torch.tensor(q).permute(0, 2, 1, 3)
    g = q.shape[2] // k.shape[2]
    tk = torch.tensor(k).permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    tv = torch.tensor(v).permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    nq, nk = q.shape[1], k.shape[1]
    mask = None
    if causal:
        mask = torch.ones(nq, nk, dtype=torch.bool).tril(diagonal=nk - nq)
    with sdpa_kernel(SDPBackend.MATH):
        o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


def check_torch_sdpa(fwd):
    for causal, (nq, nk) in itertools.product([False, True], [(33, 33), (20, 47)]):
        q, k, v = tiny_problem(B=2, Hq=6, Hkv=3, Nq=nq, Nk=nk, d=16, s=1.0)
        o, _ = fwd(q, k, v, 0.25, causal)
        np.testing.assert_allclose(o, torch_sdpa(q, k, v, 0.25, causal), rtol=0, atol=1e-12)


def check_gqa_replication(fwd):
    q, k, v = tiny_problem(B=1, Hq=6, Hkv=2, Nq=10, Nk=10, d=4)
    o, lse = fwd(q, k, v, 0.5, True)
    o2, lse2 = fwd(q, np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2), 0.5, True)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-14)


def check_key_shift_invariance(fwd):
    # adding one vector u to every key adds scale*q_i.u to the whole row i of S: O unchanged
    q, k, v = tiny_problem(B=1, Hq=2, Hkv=2, Nq=9, Nk=9, d=4)
    u = rand(4)
    for causal in (False, True):
        o1, lse1 = fwd(q, k, v, 0.5, causal)
        o2, lse2 = fwd(q, k + u, v, 0.5, causal)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        shift = 0.5 * np.einsum("bnhd,d->bhn", q, u)
        np.testing.assert_allclose(lse2 - lse1, shift, rtol=0, atol=1e-12)


def check_blockwise_invariance(fwd):
    # the online-softmax model over random key partitions equals the materialised result
    for causal, (nq, nk) in itertools.product([False, True], [(13, 13), (7, 29), (29, 17)]):
        q, k, v = tiny_problem(B=2, Hq=4, Hkv=2, Nq=nq, Nk=nk, d=5, s=3.0)
        o, lse = fwd(q, k, v, 0.7, causal)
        for _ in range(4):
            cuts = sorted(RNG.choice(np.arange(1, nk), size=RNG.integers(0, min(6, nk - 1) + 1), replace=False))
            edges = [0] + list(cuts) + [nk]
            blocks = list(zip(edges[:-1], edges[1:]))
            ob, lseb = attn_ref.blockwise_forward(q, k, v, 0.7, causal, blocks)
            np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, lseb, rtol=0, atol=1e-12)


def check_window_special_cases(fwd):
    """Sliding windows reduce to known results: (no left limit, right 0) is
    causal; no limits is the plain softmax; (0, 0) leaves each row the one
    key on its diagonal, so O_i = V[i + Nk - Nq] and LSE_i is that key's
    logit (rows whose diagonal key does not exist see nothing)."""
    for nq, nk in [(9, 9), (6, 11), (11, 6)]:
        q, k, v = tiny_problem(B=1, Hq=2, Hkv=1, Nq=nq, Nk=nk, d=4, s=1.5)
        oc, lc = fwd(q, k, v, 0.7, True)
        ow, lw = fwd(q, k, v, 0.7, False, window=(-1, 0))
        np.testing.assert_allclose(ow, oc, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lw, lc, rtol=0, atol=1e-13)
        of, lf = fwd(q, k, v, 0.7, False)
        ow, lw = fwd(q, k, v, 0.7, False, window=(-1, -1))
        np.testing.assert_array_equal(ow, of)
        np.testing.assert_array_equal(lw, lf)
        o0, l0 = fwd(q, k, v, 0.7, False, window=(0, 0))
        for i in range(nq):
            j = i + nk - nq
            for h in range(2):
                if 0 <= j < nk:
                    np.testing.assert_allclose(o0[0, i, h], v[0, j, 0], rtol=0, atol=1e-13)
                    np.testing.assert_allclose(l0[0, h, i], 0.7 * q[0, i, h] @ k[0, j, 0], rtol=0, atol=1e-13)
                else:
                    assert np.all(o0[0, i, h] == 0) and l0[0, h, i] == -np.inf


def check_window_brute_force(fwd):
    for window, causal, (nq, nk) in [((1, 0), False, (8, 8)), ((2, 3), False, (7, 12)), ((0, 2), False, (12, 7)),
                                     ((3, -1), False, (10, 10)), ((2, 5), True, (9, 9))]:
        q, k, v = tiny_problem(B=1, Hq=2, Hkv=2, Nq=nq, Nk=nk, d=3, s=1.5)
        o, lse = fwd(q, k, v, 0.8, causal, window=window)
        o_bf, lse_bf = brute_force(q, k, v, 0.8, causal, window)
        np.testing.assert_allclose(o, o_bf, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lse_bf, rtol=0, atol=1e-12)


FORWARD_PINS = [check_worked_examples, check_constant_v, check_zero_q, check_one_hot, check_causal_row0,
                check_brute_force, check_torch_sdpa, check_gqa_replication, check_key_shift_invariance,
                check_blockwise_invariance, check_window_special_cases, check_window_brute_force]


@pytest.mark.parametrize("pin", FORWARD_PINS + [check_rows_sum_to_one], ids=lambda f: f.__name__)
def test_forward_pin(pin):
    pin(attn_ref.forward)


# --------------------------------------------------------------- backward --

def loss(q, k, v, do, scale, causal, window=None):
    o, _ = attn_ref.forward(q, k, v, scale, causal, window=window)
    return float(np.sum(o * do))


def check_finite_differences(bwd):
    for causal, (nq, nk), window in [(False, (5, 5), None), (True, (6, 6), None), (True, (4, 7), None),
                                     (False, (6, 6), (1, 2)), (True, (7, 5), (2, 0))]:
        q, k, v = tiny_problem(B=1, Hq=2, Hkv=1, Nq=nq, Nk=nk, d=3, s=1.2)
        do = rand(*q.shape)
        dq, dk, dv = bwd(q, k, v, do, 0.6, causal, window=window)
        eps = 1e-6
        for x, g in ((q, dq), (k, dk), (v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + eps
                lp = loss(q, k, v, do, 0.6, causal, window)
                x[idx] = old - eps
                lm = loss(q, k, v, do, 0.6, causal, window)
                x[idx] = old
                num[idx] = (lp - lm) / (2 * eps)
            np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def check_torch_autograd(bwd):
    from torch.nn.attention import SDPBackend, sdpa_kernel
    for causal, (nq, nk) in [(False, (24, 24)), (True, (24, 24)), (True, (12, 30))]:
        q, k, v = tiny_problem(B=2, Hq=4, Hkv=2, Nq=nq, Nk=nk, d=8)
        do = rand(*q.shape)
        dq, dk, dv = bwd(q, k, v, do, 0.35, causal)
        tq = torch.tensor(q, requires_grad=True)
        tk = torch.tensor(k, requires_grad=True)
        tv = torch.tensor(v, requires_grad=True)
        g = 2
        mask = torch.ones(nq, nk, dtype=torch.bool).tril(diagonal=nk - nq) if causal else None
        with sdpa_kernel(SDPBackend.MATH):
            o = torch.nn.functional.scaled_dot_product_attention(
                tq.permute(0, 2, 1, 3), tk.permute(0, 2, 1, 3).repeat_interleave(g, 1),
                tv.permute(0, 2, 1, 3).repeat_interleave(g, 1), attn_mask=mask, scale=0.35)
        o.permute(0, 2, 1, 3).backward(torch.tensor(do))
        np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


def check_gradient_identities(bwd):
    # sum_j P_ij = 1 gives sum over keys of dV = sum over the group's queries of dO;
    # sum_j dS_ij = 0 gives sum over keys of dK = 0 (every row sees >= 1 key here).
    for causal in (False, True):
        q, k, v = tiny_problem(B=2, Hq=4, Hkv=2, Nq=11, Nk=11, d=4)
        do = rand(*q.shape)
        dq, dk, dv = bwd(q, k, v, do, 0.5, causal)
        want_dv = do.reshape(2, 11, 2, 2, 4).sum(axis=(1, 3))
        np.testing.assert_allclose(dv.sum(axis=1), want_dv, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk.sum(axis=1), 0.0, rtol=0, atol=1e-12)
        if causal:
            np.testing.assert_allclose(dq[:, 0], 0.0, rtol=0, atol=1e-12)  # row 0 sees one key


def check_constant_v_grads(bwd):
    q, k, _ = tiny_problem(B=1, Hq=2, Hkv=1, Nq=7, Nk=7, d=3)
    v = np.broadcast_to(rand(3), k.shape).copy()
    do = rand(*q.shape)
    dq, dk, _ = bwd(q, k, v, do, 0.5, True)
    np.testing.assert_allclose(dq, 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, 0.0, rtol=0, atol=1e-12)


def check_gqa_grad_group_sum(bwd):
    q, k, v = tiny_problem(B=1, Hq=6, Hkv=2, Nq=8, Nk=8, d=4)
    do = rand(*q.shape)
    dq, dk, dv = bwd(q, k, v, do, 0.5, True)
    dq2, dk2, dv2 = bwd(q, np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2), do, 0.5, True)
    np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(1, 8, 2, 3, 4).sum(axis=3), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(1, 8, 2, 3, 4).sum(axis=3), rtol=0, atol=1e-13)


BACKWARD_PINS = [check_finite_differences, check_torch_autograd, check_gradient_identities, check_constant_v_grads,
                 check_gqa_grad_group_sum]


@pytest.mark.parametrize("pin", BACKWARD_PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin):
    pin(attn_ref.backward)


def test_empty_rows():
    # causal with Nq > Nk, bottom-right: the first Nq - Nk rows see no key
    q, k, v = tiny_problem(B=1, Hq=2, Hkv=2, Nq=6, Nk=3, d=2)
    o, lse = attn_ref.forward(q, k, v, 0.5, True)
    assert np.all(o[:, :3] == 0) and np.all(np.isneginf(lse[:, :, :3]))
    assert np.all(np.isfinite(lse[:, :, 3:]))
    do = rand(*q.shape)
    dq, dk, dv = attn_ref.backward(q, k, v, do, 0.5, True)
    assert np.all(dq[:, :3] == 0)
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def test_rows_subset_matches_full():
    q, k, v = tiny_problem(B=1, Hq=2, Hkv=1, Nq=40, Nk=40, d=4)
    o, lse = attn_ref.forward(q, k, v, 0.5, True)
    rows = np.array([0, 3, 17, 39])
    o2, lse2 = attn_ref.forward(q, k, v, 0.5, True, rows=rows)
    np.testing.assert_array_equal(o[:, rows], o2)
    np.testing.assert_array_equal(lse[:, :, rows], lse2)


# ------------------------------------------------------ planted mistakes --

def _fails_some(pins, fn):
    failed = []
    for pin in pins:
        try:
            pin(fn)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


MUTANTS = {
    "scale_dropped": ("_scores", lambda orig: (
        lambda Q, K, scale, rows, nq, causal, window=None: orig(Q, K, 1.0, rows, nq, causal, window))),
    "top_left_causal": ("visible_mask", lambda orig: (
        lambda rows, nq, nk, causal, window=None: orig(rows, nk, nk, causal, window))),
    "mask_off_by_one": ("visible_mask", lambda orig: (
        lambda rows, nq, nk, causal, window=None: orig(np.asarray(rows) - 1, nq, nk, causal, window))),
    "window_left_off_by_one": ("visible_mask", lambda orig: (
        lambda rows, nq, nk, causal, window=None: orig(
            rows, nq, nk, causal, None if window is None else (window[0] + 1 if window[0] >= 0 else -1, window[1])))),
    "window_right_ignored": ("visible_mask", lambda orig: (
        lambda rows, nq, nk, causal, window=None: orig(
            rows, nq, nk, causal, None if window is None else (window[0], -1)))),
    "lse_log2": ("_softmax_stats", lambda orig: (
        lambda S: (lambda P, l: (P, l / math.log(2)))(*orig(S)))),
    "softmax_not_normalised": ("_softmax_stats", lambda orig: (
        lambda S: (lambda P, l: (P * np.exp(l)[:, None] / np.exp(S.max(axis=1))[:, None], l))(*orig(S)))),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_forward_mistake_is_caught(name, monkeypatch):
    attr, make = MUTANTS[name]
    monkeypatch.setattr(attn_ref, attr, make(getattr(attn_ref, attr)))
    failed = _fails_some(FORWARD_PINS, attn_ref.forward)
    assert failed, f"mutant {name} passed every forward pin"


BWD_MUTANTS = {
    "ds_sign": lambda orig: (lambda P, dP, D: P * (dP + D[:, None])),
    "ds_drops_D": lambda orig: (lambda P, dP, D: P * dP),
    "ds_transposed_P": lambda orig: (lambda P, dP, D: (P.T if P.shape[0] == P.shape[1] else P) * (dP - D[:, None])),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_planted_backward_mistake_is_caught(name, monkeypatch):
    monkeypatch.setattr(attn_ref, "_softmax_grad", BWD_MUTANTS[name](attn_ref._softmax_grad))
    failed = _fails_some(BACKWARD_PINS, attn_ref.backward)
    assert failed, f"mutant {name} passed every backward pin"


def test_zero_scale_weights_visible_keys_equally():
    """scale = 0: O_i is the mean of the visible V rows and LSE_i = ln(count)."""
    rng = np.random.default_rng(41)
    q, k, v = (rng.normal(size=(1, n, 2, 16)) for n in (7, 9, 9))
    for causal in (False, True):
        o, lse = attn_ref.forward(q, k, v, 0.0, causal)
        off = 9 - 7
        for i in range(7):
            cnt = (i + off + 1) if causal else 9
            np.testing.assert_allclose(o[0, i], v[0, :cnt].mean(axis=0), atol=1e-12)
            np.testing.assert_allclose(lse[0, :, i], np.log(cnt), atol=1e-12)


def test_negative_scale_is_positive_scale_with_negated_keys():
    """softmax(-c Q K^T) = softmax(c Q (-K)^T): the row max must be that of
    the scaled scores, not of the raw ones."""
    rng = np.random.default_rng(42)
    q, k, v = (rng.normal(size=(1, 11, 2, 8)) * 3 for _ in range(3))
    for causal in (False, True):
        o1, l1 = attn_ref.forward(q, k, v, -0.7, causal)
        o2, l2 = attn_ref.forward(q, -k, v, 0.7, causal)
        np.testing.assert_allclose(o1, o2, atol=1e-12)
        np.testing.assert_allclose(l1, l2, atol=1e-12)
        # against a scalar loop
        for i in (0, 5, 10):
            s = [-0.7 * float(q[0, i, 1] @ k[0, j, 1]) for j in range(11) if not causal or j <= i]
            m = max(s)
            w = [math.exp(t - m) for t in s]
            ref = sum(wj * v[0, j, 1] for j, wj in enumerate(w)) / sum(w)
            np.testing.assert_allclose(o1[0, i, 1], ref, atol=1e-12)


def brute_abs_terms(q, k, v, do, scale, causal):
    """backward_abs_terms by scalar loops (math.fsum), with D_i formed as
    sum_j P_ij dP_ij (equal to sum_c dO_ic O_ic in exact arithmetic)."""
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    g = Hq // Hkv
    a_dq, a_dk, a_dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            for i in range(Nq):
                keys = [j for j in range(Nk) if seen(i, j, Nq, Nk, causal, None)]
                if not keys:
                    continue
                logits = [scale * math.fsum(q[b, i, h, c] * k[b, j, kv, c] for c in range(d)) for j in keys]
                top = max(logits)
                w = [math.exp(s - top) for s in logits]
                tot = math.fsum(w)
                P = [x / tot for x in w]
                dP = [math.fsum(do[b, i, h, c] * v[b, j, kv, c] for c in range(d)) for j in keys]
                D = math.fsum(p * dp for p, dp in zip(P, dP))
                dS = [abs(p * (dp - D)) for p, dp in zip(P, dP)]
                for c in range(d):
                    a_dq[b, i, h, c] = scale * math.fsum(s * abs(k[b, j, kv, c]) for s, j in zip(dS, keys))
                for t, j in enumerate(keys):
                    for c in range(d):
                        a_dk[b, j, kv, c] += scale * dS[t] * abs(q[b, i, h, c])
                        a_dv[b, j, kv, c] += P[t] * abs(do[b, i, h, c])
    return a_dq, a_dk, a_dv


@pytest.mark.parametrize("causal", [False, True])
def test_backward_abs_terms_brute_force(causal):
    rng = np.random.default_rng(12)
    B, Hq, Hkv, N, d = 1, 4, 2, 9, 5
    q, k, v, do = (rng.normal(size=(B, N, h, d)) * 1.5 for h in (Hq, Hkv, Hkv, Hq))
    got = attn_ref.backward_abs_terms(q, k, v, do, 0.7, causal)
    want = brute_abs_terms(q, k, v, do, 0.7, causal)
    for g_, w_ in zip(got, want):
        np.testing.assert_allclose(g_, w_, rtol=1e-10, atol=1e-12)


def test_backward_abs_terms_bound_a_perturbed_ds():
    """Rounding each dS_ij (P_ij) with relative error up to e moves dQ, dK
    (dV) by at most e times the terms: checked on a direct fp64 computation
    with random perturbations of the largest allowed size."""
    rng = np.random.default_rng(13)
    N, d, scale, e = 12, 6, 0.5, 2.0 ** -8
    q, k, v, do = (rng.normal(size=(1, N, 1, d)) * 2.0 for _ in range(4))
    a_dq, a_dk, a_dv = attn_ref.backward_abs_terms(q, k, v, do, scale, True)
    Q, K, V, dO = q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0]
    P = attn_ref.probabilities(Q, K, scale, True)
    dP = dO @ V.T
    dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
    for _ in range(20):
        eps = e * rng.choice([-1.0, 1.0], size=dS.shape)
        dS2, P2 = dS * (1 + eps), P * (1 + eps)
        assert np.all(np.abs(scale * (dS2 - dS) @ K) <= e * a_dq[0, :, 0] + 1e-12)
        assert np.all(np.abs(scale * (dS2 - dS).T @ Q) <= e * a_dk[0, :, 0] + 1e-12)
        assert np.all(np.abs((P2 - P).T @ dO) <= e * a_dv[0, :, 0] + 1e-12)
