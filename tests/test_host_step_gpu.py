"""fa_step_host: forward + backward on host buffers, pipelined over the
batch (inputs in on one copy stream, compute on a library stream, results
out on another; a one-element batch is cut into two halves of its kv
heads; the forward runs over two groups of these chunks, uneven for an odd
count, the backward over all of them at once). Checked through the C ABI element by element
against the fp64 oracle (O, LSE within the parity tolerances; dQ, dK, dV
within them plus half a bf16 ulp of the value, as these GQA gradients
exceed |x| = 4),
and against fa_fwd + fa_bwd on device buffers for the same inputs: O and LSE
bit for bit (each row is computed by the same kernel either way), the
gradients within the backward's tolerance (dQ is summed in fp32 in a
nondeterministic order)."""
import math

import pytest
import torch

import workloads
from oracle import attn_ref
from tests.gpu_util import assert_close, assert_close_scaled, assert_lse, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_99_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    m.fa_debug_set(0, 0)
    return m


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal
    (3, 4, 2, 300, 300, 128, True),
    (2, 2, 2, 200, 520, 64, False),
    (1, 4, 4, 256, 256, 128, False),  # one batch element: two chunks of two kv heads (2-D copies)
    (1, 8, 2, 300, 420, 128, True),   # one batch element, GQA: two chunks of one kv head and four query heads
    (1, 3, 3, 129, 129, 64, True),    # odd Hkv: one chunk
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("pinned", [True, False])
def test_step_host_matches_device_calls(fa, case, pinned):
    B, Hq, Hkv, Nq, Nk, d, causal = case
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=B * 100 + Nq, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    args = (B, Hq, Hkv, Nq, Nk, d, scale, int(causal))
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = torch.empty_like(q), torch.empty((B, Hq, Nq), device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert fa.fa_fwd(q, k, v, o, lse, *args) == 0
    assert fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, *args) == 0

    host = {n: (x[n].pin_memory() if pinned else x[n].clone()) for n in ("q", "k", "v", "do")}
    outs = {n: torch.full(t.shape, float("nan"), dtype=t.dtype, pin_memory=pinned)
            for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    st = fa.fa_step_host(host["q"], host["k"], host["v"], host["do"], outs["o"], outs["lse"], outs["dq"], outs["dk"],
                         outs["dv"], *args)
    assert st == 0
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    assert torch.equal(outs["o"], o.cpu())
    assert torch.equal(outs["lse"], lse.cpu())
    for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
        got = outs[name]
        assert torch.isfinite(got.float()).all(), name
        assert_close(name, to64(got), to64(ref.cpu()))
    # the oracle, element by element, on the host results
    xs = [x[n].double().numpy() for n in ("q", "k", "v", "do")]
    ro, rlse = attn_ref.forward(*xs[:3], scale, causal)
    assert_close("o vs oracle", to64(outs["o"]), ro)
    assert_lse(to64(outs["lse"]), rlse)
    # gradients of these GQA cases reach |x| > 4 (dV of the first keys sums
    # over every query of the group), where output rounding alone can pass
    # 2e-2: the bound grows with the value (assert_close_scaled)
    for name, ref in zip(("dq", "dk", "dv"), attn_ref.backward(*xs, scale, causal)):
        assert_close_scaled(f"{name} vs oracle", to64(outs[name]), ref)


def test_step_host_back_to_back(fa):
    """Consecutive calls overlap (the inputs of one call are copied in while
    the previous one computes, and its kernels run while the previous one's
    results go out; the device buffers alternate between calls):
    three calls enqueued without a synchronisation in between, each on its
    own inputs and outputs, so that the third reuses the first one's device
    buffer, all match the device calls on their inputs."""
    B, Hq, Hkv, Nq, Nk, d, causal = 1, 8, 2, 700, 700, 128, True
    args = (B, Hq, Hkv, Nq, Nk, d, 1.0 / math.sqrt(d), int(causal))
    runs = []
    for seed in (11, 12, 13):
        x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=seed, with_dout=True)
        host = {n: x[n].pin_memory() for n in ("q", "k", "v", "do")}
        outs = {n: torch.full(s, float("nan"), dtype=t, pin_memory=True)
                for n, s, t in (("o", (B, Nq, Hq, d), torch.bfloat16), ("lse", (B, Hq, Nq), torch.float32),
                                ("dq", (B, Nq, Hq, d), torch.bfloat16), ("dk", (B, Nk, Hkv, d), torch.bfloat16),
                                ("dv", (B, Nk, Hkv, d), torch.bfloat16))}
        runs.append((x, host, outs))
    torch.cuda.synchronize()
    for x, host, outs in runs:
        assert fa.fa_step_host(host["q"], host["k"], host["v"], host["do"], outs["o"], outs["lse"], outs["dq"],
                               outs["dk"], outs["dv"], *args) == 0
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    for x, host, outs in runs:
        q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
        o, lse = torch.empty_like(q), torch.empty((B, Hq, Nq), device="cuda", dtype=torch.float32)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        assert fa.fa_fwd(q, k, v, o, lse, *args) == 0
        assert fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, *args) == 0
        torch.cuda.synchronize()
        assert torch.equal(outs["o"], o.cpu())
        assert torch.equal(outs["lse"], lse.cpu())
        for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
            assert_close(name, to64(outs[name]), to64(ref.cpu()))


def test_step_host_stream_ordered_after_call(fa):
    """The kernels run on a library stream, but the caller's stream is
    ordered after every copy and kernel of the call: synchronising that
    stream alone (not the device) is enough to read the host results, and
    work enqueued on it afterwards sees them. Two calls on a side stream,
    the second enqueued right after the first."""
    B, Hq, Hkv, Nq, Nk, d, causal = 1, 8, 2, 1000, 1000, 128, True
    args = (B, Hq, Hkv, Nq, Nk, d, 1.0 / math.sqrt(d), int(causal))
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed=21, with_dout=True)
    host = {n: x[n].pin_memory() for n in ("q", "k", "v", "do")}
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = torch.empty_like(q), torch.empty((B, Hq, Nq), device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert fa.fa_fwd(q, k, v, o, lse, *args) == 0
    assert fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, *args) == 0
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    outs = []
    for _ in range(2):
        outs.append({n: torch.full(t.shape, float("nan"), dtype=t.dtype, pin_memory=True)
                     for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))})
        assert fa.fa_step_host(host["q"], host["k"], host["v"], host["do"], outs[-1]["o"], outs[-1]["lse"],
                               outs[-1]["dq"], outs[-1]["dk"], outs[-1]["dv"], *args, stream=side) == 0
    # a device copy of the second call's dK enqueued on the side stream
    with torch.cuda.stream(side):
        dk_dev = torch.empty_like(dk)
        dk_dev.copy_(outs[1]["dk"], non_blocking=True)
    side.synchronize()
    for out in outs:
        assert torch.equal(out["o"], o.cpu())
        assert torch.equal(out["lse"], lse.cpu())
        for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
            assert_close(name, to64(out[name]), to64(ref.cpu()))
    assert torch.equal(dk_dev.cpu(), outs[1]["dk"])
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
