"""fa_bwd_noalloc: the backward pass for callers that may not allocate
device memory during the call (serving loops with a fixed memory plan, code
that runs where the CUDA allocator must not be entered). Its workspace is a
fixed device array inside the library instead of a per-call allocation.

Checked through the C ABI against fa_bwd on two calls in a row with
different problems, so a result that depended on what an earlier call left
in the shared array would show. Kept in a file that pytest collects last."""
import math

import pytest
import torch

import workloads
from tests.gpu_util import assert_close, to64

pytestmark = pytest.mark.gpu

FA_ERR_UNSUPPORTED = 2


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_99_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    m.fa_debug_set(0, 0)
    return m


def both_paths(fa, B, Hq, Hkv, Nq, Nk, d, causal, seed):
    x = workloads.make_inputs(B, Hq, Hkv, Nq, Nk, d, seed, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    args = (B, Hq, Hkv, Nq, Nk, d, scale, int(causal))
    ref = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    assert fa.fa_bwd(q, k, v, o, lse, do, *ref, *args) == 0
    got = [torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))]
    assert fa.fa_bwd_noalloc(q, k, v, o, lse, do, *got, *args) == 0
    torch.cuda.synchronize()
    assert fa.fa_get_status() == 0
    return got, ref


def test_noalloc_matches_fa_bwd_twice(fa):
    cases = [
        (1, 4, 2, 300, 300, 128, True, 31),   # GQA, causal, ragged length
        (2, 2, 2, 200, 520, 64, False, 32),   # another shape: must not depend on the previous contents
    ]
    for B, Hq, Hkv, Nq, Nk, d, causal, seed in cases:
        got, ref = both_paths(fa, B, Hq, Hkv, Nq, Nk, d, causal, seed)
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(g).all(), name
            assert_close(name, to64(g), to64(r))


def test_noalloc_rejects_workspace_beyond_the_array(fa):
    # 4 * B*Hq*Nq*(d + 2) bytes = 4 * 16*16384*130 > 64 MiB
    B, Hq, Hkv, N, d = 1, 16, 16, 16384, 128
    p = 1 << 20  # aligned, non-null: the size check fails before anything is launched
    assert fa.fa_bwd_noalloc(*([p] * 9), B, Hq, Hkv, N, N, d, d ** -0.5, 1) == FA_ERR_UNSUPPORTED
    assert fa.fa_get_status() == 0
