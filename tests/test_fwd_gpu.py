"""Forward parity on a GB300: the CUDA path (through the C ABI) against the
fp64 CPU oracle on identical seeded bf16 inputs."""
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
    return m


def run_case(fa, B, Hq, Hkv, Nq, Nk, d, causal, seed, sigma_qk=1.0, rows=None):
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed, sigma_qk=sigma_qk)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    qn, kn, vn = (x[n].double().numpy() for n in ("q", "k", "v"))
    ro, rlse = attn_ref.forward(qn, kn, vn, scale, causal, rows=rows)
    go, glse = to64(o), to64(lse)
    if rows is not None:
        go, glse = go[:, rows], glse[:, :, rows]
    assert_close("o", go, ro)
    assert_lse(glse, rlse)
    return o, lse


SMALL = [
    # B, Hq, Hkv, Nq, Nk, d
    (1, 2, 2, 1, 1, 64),
    (1, 2, 1, 17, 17, 128),
    (2, 3, 3, 128, 128, 64),
    (1, 4, 2, 129, 129, 128),
    (1, 2, 2, 255, 255, 64),
    (2, 2, 2, 256, 256, 128),
    (1, 4, 1, 300, 300, 128),
    (1, 2, 2, 513, 513, 64),
    (1, 2, 2, 100, 700, 128),   # Nq < Nk
    (1, 2, 2, 700, 100, 128),   # Nq > Nk: causal rows with no visible key
    (1, 1, 1, 1, 1000, 64),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(fa, shape, causal):
    B, Hq, Hkv, Nq, Nk, d = shape
    run_case(fa, B, Hq, Hkv, Nq, Nk, d, causal, seed=hash((shape, causal)) % 10000)


def split_plan(n_sms, B, Hq, Nq, causal):
    """Which units the forward runs as two single-stage (128-row) items: the
    T = units mod SMs units of the last, partly filled round, when 2T <= SMs
    (non-causal, Nq > 128 only). Returns T, or 0 for no split."""
    units = B * Hq * ((Nq + 255) // 256)
    t = units % n_sms
    return t if (t and 2 * t <= n_sms and not causal and Nq > 128) else 0


SPLIT = [
    # B, Hq, Hkv, Nq, Nk, d, units split on a 152-SM GB300
    (1, 2, 2, 300, 700, 128, 4),    # ragged Nq (the last unit holds 44 rows, all in its first half) and Nk
    (1, 40, 40, 256, 1000, 64, 40),
    (1, 54, 6, 768, 640, 128, 10),  # 162 units: a full round, then 10 split units (GQA)
    (2, 36, 4, 512, 384, 128, 0),   # 144 units: more than half the SMs, no split
    (1, 2, 2, 128, 384, 64, 0),     # one 128-row block: nothing to split
]


@pytest.mark.parametrize("shape", SPLIT, ids=lambda s: "x".join(map(str, s)))
def test_row_split_tail(fa, shape):
    """Non-causal units of the last round run as one item per 128-row stage;
    parity against the oracle with and without that split."""
    B, Hq, Hkv, Nq, Nk, d, t152 = shape
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    if n_sms == 152:
        assert split_plan(n_sms, B, Hq, Nq, False) == t152
    run_case(fa, B, Hq, Hkv, Nq, Nk, d, False, seed=sum(shape))


def test_workload_small_full(fa):
    w = workloads.WORKLOADS[0]
    run_case(fa, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.causal, w.seed, w.sigma_qk)


def last_round_heads(n_sms, B, Hq, Nq, causal):
    """(batch, head) pairs with a work item in the forward's last scheduling
    round: non-causal units run head by head (query blocks of one head in a
    row), the last round's units split by rows; causal rounds cover every
    head (longest query blocks first, so the last round holds block 0s)."""
    mblocks = (Nq + 255) // 256
    units = B * Hq * mblocks
    if causal:
        return {(b, h) for b in range(B) for h in range(Hq)}
    t = split_plan(n_sms, B, Hq, Nq, causal)
    full = units - t
    n_items = full + 2 * t
    first_last = (n_items - 1) // n_sms * n_sms  # first item of the last round
    heads = set()
    for item in range(first_last, n_items):
        u = item if item < full else full + (item - full) // 2
        bh = u // mblocks
        heads.add((bh // Hq, bh % Hq))
    return heads


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_workload_full_size_whole_heads(fa, idx):
    """Full-size run in the benchmark's launch configuration; the oracle
    checks every row of two whole heads, the first (batch, head) and the
    last, which runs in the last scheduling round, and sampled rows of a
    third head."""
    w = workloads.WORKLOADS[idx]
    x = workloads.workload_inputs(w)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    last = (w.B - 1, w.Hq - 1)
    assert last in last_round_heads(n_sms, w.B, w.Hq, w.Nq, w.causal)
    go, glse = to64(o), to64(lse)
    rng = np.random.default_rng(w.seed)
    sampled = np.unique(np.concatenate([rng.choice(w.Nq, 96, replace=False), [0, 1, 127, 128, 255, w.Nq - 1]]))
    for (b, h), rows in (((0, 0), None), (last, None), ((w.B // 2, w.Hq // 2), sampled)):
        kv = h // (w.Hq // w.Hkv)
        qn = x["q"][b:b + 1, :, h:h + 1].double().numpy()
        kn = x["k"][b:b + 1, :, kv:kv + 1].double().numpy()
        vn = x["v"][b:b + 1, :, kv:kv + 1].double().numpy()
        ro, rlse = attn_ref.forward(qn, kn, vn, w.scale, w.causal, rows=rows)
        sel = slice(None) if rows is None else rows
        assert_close(f"o[b{b},h{h}]", go[b:b + 1, sel, h:h + 1], ro)
        assert_lse(glse[b:b + 1, h:h + 1, sel], rlse)
    # properties that hold at any size
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_constant_v_identity(fa):
    B, H, N, d = 1, 2, 333, 128
    x = workloads.make_inputs(B, H, H, N, N, d, seed=5, sigma_qk=2.0)
    v0 = torch.randn(d).to(torch.bfloat16)
    v = v0.expand(B, N, H, d).contiguous()
    for causal in (False, True):
        o, _ = fa.forward(x["q"].cuda(), x["k"].cuda(), v.cuda(), causal=causal)
        torch.cuda.synchronize()
        err = (o.double().cpu() - v0.double().expand(B, N, H, d)).abs().max().item()
        assert err <= 2e-2, err


def test_zero_q_mean(fa):
    B, H, N, d = 1, 2, 260, 64
    x = workloads.make_inputs(B, H, H, N, N, d, seed=6)
    q = torch.zeros_like(x["q"])
    o, lse = fa.forward(q.cuda(), x["k"].cuda(), x["v"].cuda(), causal=True)
    torch.cuda.synchronize()
    vc = x["v"].double().cumsum(dim=1) / torch.arange(1, N + 1, dtype=torch.float64)[None, :, None, None]
    assert (o.double().cpu() - vc).abs().max().item() <= 2e-2
    want = torch.log(torch.arange(1, N + 1, dtype=torch.float64))
    assert (lse.double().cpu() - want[None, None]).abs().max().item() <= 1e-3


@pytest.mark.parametrize("causal", [True, False])  # non-causal: 16 units, each run as two 128-row items
def test_deterministic_and_offset_invariant(fa, causal):
    B, Hq, Hkv, N, d = 2, 4, 2, 384, 128
    x = workloads.make_inputs(B, Hq, Hkv, N, N, d, seed=9)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = fa.forward(q, k, v, causal=causal)
    o2, l2 = fa.forward(q, k, v, causal=causal)
    # same tensors placed at a 16-byte-aligned offset inside larger buffers
    pad = 8
    bufs = []
    for t in (q, k, v):
        big = torch.empty(t.numel() + pad, dtype=t.dtype, device=t.device)
        big[pad:].copy_(t.reshape(-1))
        bufs.append(big[pad:].view(t.shape))
    o3, l3 = fa.forward(*bufs, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_memory_linear_in_n(fa):
    """The score matrix never reaches device memory: a forward + backward at
    N = 16384 (one head, d = 64) may take the O(N) workspace of the backward
    (4 * Nq * (d + 2) bytes per head, about 4 MB here) but nothing near the
    N^2 * 4 bytes = 1 GiB a materialised S would need."""
    N, d = 16384, 64
    x = workloads.make_inputs(1, 1, 1, N, N, d, seed=5, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = torch.empty_like(q), torch.empty((1, 1, N), device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    args = (1, 1, 1, N, N, d, d ** -0.5, 1)
    # once at a small size first: loading the library's device code and its
    # fixed arrays (the 64 MiB scratch of fa_bwd_noalloc) is not part of a call
    small = (1, 1, 1, 256, 256, d, d ** -0.5, 1)
    assert fa.fa_fwd(q, k, v, o, lse, *small) == 0
    assert fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, *small) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert fa.fa_fwd(q, k, v, o, lse, *args) == 0
    assert fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, *args) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert fa.fa_get_status() == 0
    assert free0 - free1 < 64 << 20, (free0 - free1)


def test_bounded_wait_reports_timeout(fa):
    """The producer withholds one tile; the consumer's bounded wait must run
    out, the kernel must exit and report FA_ERR_TIMEOUT, and the context must
    stay usable."""
    B, H, N, d = 1, 1, 256, 64
    x = workloads.make_inputs(B, H, H, N, N, d, seed=11)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    assert fa.fa_get_status() == 0
    assert fa.fa_debug_set(20_000_000, 1) == 0
    try:
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
        assert fa.fa_fwd(q, k, v, o, lse, B, H, H, N, N, d, d ** -0.5, 0) == 0
        assert fa.fa_get_status() == 5
    finally:
        fa.fa_debug_set(0, 0)
    run_case(fa, B, H, H, N, N, d, False, seed=11)


def test_debug_exp2(fa):
    x = torch.linspace(-130.0, 0.0, 1 << 16, device="cuda", dtype=torch.float32)
    want = torch.exp2(x.double())
    for mode in (0, 1):
        y = torch.empty_like(x)
        assert fa.fa_debug_exp2(x, y, x.numel(), mode) == 0
        torch.cuda.synchronize()
        ok = x > -126
        rel = ((y.double() - want) / want)[ok].abs()
        assert rel.max().item() < (2e-6 if mode == 0 else 1e-4), (mode, rel.max().item())
        assert y[x <= -127.5].abs().max().item() < 1e-37


WINDOWS = [
    # B, Hq, Hkv, Nq, Nk, d, (left, right)
    (1, 2, 2, 300, 300, 128, (64, 0)),      # causal local window narrower than a tile
    (1, 2, 1, 700, 700, 64, (200, 0)),
    (1, 2, 2, 513, 513, 128, (128, 128)),   # symmetric, ragged length
    (1, 2, 2, 400, 900, 128, (300, 50)),    # Nq < Nk
    (1, 2, 2, 900, 400, 128, (100, 0)),     # Nq > Nk: rows with no visible key
    (2, 4, 2, 1024, 1024, 128, (0, 0)),     # one key per row
    (1, 2, 2, 600, 600, 64, (-1, 300)),     # right bound only
    (1, 2, 2, 256, 256, 128, (1000, 1000)), # a window covering every key
    (1, 3, 3, 1000, 1000, 128, (500, -1)),  # left bound only
]


@pytest.mark.parametrize("shape", WINDOWS, ids=lambda s: "x".join(map(str, s[:6])) + f"-w{s[6][0]}_{s[6][1]}")
def test_window(fa, shape):
    B, Hq, Hkv, Nq, Nk, d, window = shape
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape[:6]) + 7 * window[0] + window[1])
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, scale=scale, window=window)
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    ro, rlse = attn_ref.forward(*(x[n].double().numpy() for n in ("q", "k", "v")), scale, False, window=window)
    assert_close("o", to64(o), ro)
    assert_lse(to64(lse), rlse)


def test_window_causal_matches_causal(fa):
    """window (no left limit, right 0) is the causal mask: the same kernel
    path and the same bits as fa_fwd with causal = 1."""
    B, Hq, Hkv, N, d = 1, 4, 2, 777, 128
    x = workloads.make_inputs(B, Hq, Hkv, N, N, d, seed=41)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = fa.forward(q, k, v, causal=True)
    o2, l2 = fa.forward(q, k, v, window=(-1, 0))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_window_full_size_sampled(fa):
    """A causal local window of 1024 keys at N = 8192 (B=2, H=16): the key
    tiles outside the window are skipped; sampled rows of two heads against
    the oracle, and every output finite."""
    B, H, N, d, window = 2, 16, 8192, 128, (1023, 0)
    x = workloads.make_inputs(B, H, H, N, N, d, seed=42)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, window=window)
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rows = np.array([0, 1, 127, 128, 1000, 1023, 1024, 1025, 4095, 4096, 8190, 8191])
    for b, h in [(0, 0), (1, 15)]:
        sl = lambda t: t[b:b + 1, :, h:h + 1].double().numpy()
        ro, rlse = attn_ref.forward(sl(x["q"]), sl(x["k"]), sl(x["v"]), d ** -0.5, False, rows=rows, window=window)
        assert_close(f"o[b{b},h{h}]", to64(o[b:b + 1, rows, h:h + 1]), ro)
        assert_lse(to64(lse[b:b + 1, h:h + 1, rows]), rlse)
