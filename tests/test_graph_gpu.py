"""The passes inside a CUDA graph: fa_fwd and fa_bwd (and their windowed
and allocation-free forms) are captured on a stream once and replayed with
new inputs copied into the captured buffers; results equal the eager calls
(bit for bit where the eager result is deterministic)."""
import math

import pytest
import torch

import workloads
from tests.gpu_util import assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_99_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    m.fa_debug_set(0, 0)
    return m


@pytest.mark.parametrize("mode", ["causal", "full", "window", "noalloc"])
def test_fwd_bwd_graph_replay(fa, mode):
    B, Hq, Hkv, N, d = 2, 8, 2, 1000, 128
    causal = mode == "causal"
    window = (300, 0) if mode == "window" else None
    scale = 1.0 / math.sqrt(d)
    xs = [workloads.make_inputs(B, Hq, Hkv, N, N, d, seed=60 + i, with_dout=True) for i in range(2)]
    # static buffers the graph reads and writes
    q, k, v, do = (xs[0][n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = torch.empty_like(q), torch.empty((B, Hq, N), device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    a = (B, Hq, Hkv, N, N, d, scale)

    def step():
        if window is not None:
            assert fa.fa_fwd_window(q, k, v, o, lse, *a, *window) == 0
            assert fa.fa_bwd_window(q, k, v, o, lse, do, dq, dk, dv, *a, *window) == 0
        else:
            assert fa.fa_fwd(q, k, v, o, lse, *a, int(causal)) == 0
            bwd = fa.fa_bwd_noalloc if mode == "noalloc" else fa.fa_bwd
            assert bwd(q, k, v, o, lse, do, dq, dk, dv, *a, int(causal)) == 0

    step()  # eager warm-up (first calls set up per-device state outside the capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for x in xs:
        for t, n in ((q, "q"), (k, "k"), (v, "v"), (do, "do")):
            t.copy_(x[n].cuda())
        g.replay()
        torch.cuda.synchronize()
        assert fa.fa_get_status() == 0
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        step()  # eager on the same inputs
        torch.cuda.synchronize()
        ref = (o, lse, dq, dk, dv)
        for name, gt, rt in zip(("o", "lse", "dk", "dv"), (got[0], got[1], got[3], got[4]),
                                (ref[0], ref[1], ref[3], ref[4])):
            assert torch.equal(gt, rt), name
        assert_close("dq", to64(got[2]), to64(ref[2]))  # dQ sums in arbitrary order
