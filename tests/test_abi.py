"""Host-only checks of the C ABI: the library builds, loads without a GPU,
exports every function include/fa.h declares, and rejects bad arguments on
the host before any device work (no GPU needed, nothing is launched)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_99_gb300 as m
    m.lib()
    return m


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(fa_\w+)\s*\(", text, flags=re.M))
    return names


def test_header_exports(fa):
    names = declared_functions()
    assert {"fa_fwd", "fa_bwd", "fa_get_status", "fa_status_string"} <= names
    L = ctypes.CDLL(fa.LIB_PATH)
    for n in sorted(names):
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_status_strings(fa):
    for code, name in fa.STATUS.items():
        assert fa.fa_status_string(code) == name
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


GOOD = dict(B=1, Hq=4, Hkv=2, Nq=64, Nk=64, d=128, scale=0.125, causal=1)
P16 = 1 << 20  # any 16-byte aligned non-null address: validation fails before it is touched


def fwd(fa, ptrs=(P16,) * 5, **kw):
    a = dict(GOOD, **kw)
    return fa.fa_fwd(*ptrs, a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"], 0)


def bwd(fa, ptrs=(P16,) * 9, **kw):
    a = dict(GOOD, **kw)
    return fa.fa_bwd(*ptrs, a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"], 0)


@pytest.mark.parametrize("call", [fwd, bwd])
@pytest.mark.parametrize("bad,code", [
    (dict(d=96), 2), (dict(d=256), 2), (dict(d=0), 1), (dict(Hq=3, Hkv=2), 1), (dict(B=0), 1),
    (dict(Nq=0), 1), (dict(Nk=-5), 1), (dict(Hkv=0), 1), (dict(causal=2), 1),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1), (dict(scale=float("-inf")), 1),
    (dict(Nq=1 << 29), 2),
])
def test_bad_sizes_rejected_on_host(fa, call, bad, code):
    assert call(fa, **bad) == code


def fwd8(fa, ptrs=(P16,) * 5, incoherent=1, **kw):
    a = dict(GOOD, **kw)
    return fa.fa_fwd_fp8(*ptrs, a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"],
                         incoherent, 0)


@pytest.mark.parametrize("bad,code", [
    (dict(d=64), 2), (dict(d=96), 2), (dict(Hq=3, Hkv=2), 1), (dict(Nq=0), 1), (dict(causal=2), 1),
    (dict(scale=float("nan")), 1), (dict(incoherent=2), 1), (dict(incoherent=-1), 1),
])
def test_fp8_bad_arguments_rejected_on_host(fa, bad, code):
    assert fwd8(fa, **bad) == code
    for which in range(5):
        ptrs = [P16] * 5
        ptrs[which] = P16 + 4
        assert fwd8(fa, ptrs=tuple(ptrs)) == 1


def step_host(fa, ptrs=(P16,) * 9, **kw):
    a = dict(GOOD, **kw)
    return fa.fa_step_host(*ptrs, a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"], 0)


def test_step_host_rejects_bad_arguments(fa):
    for which in range(9):
        ptrs = [P16] * 9
        ptrs[which] = 0
        assert step_host(fa, ptrs=tuple(ptrs)) == 1
    assert step_host(fa, d=96) == 2
    assert step_host(fa, Hq=3, Hkv=2) == 1
    assert step_host(fa, Nq=0) == 1


@pytest.mark.parametrize("which", range(5))
def test_bad_pointers_fwd(fa, which):
    for bad in (0, P16 + 8):  # null, misaligned
        ptrs = [P16] * 5
        ptrs[which] = bad
        assert fwd(fa, ptrs=tuple(ptrs)) == 1


@pytest.mark.parametrize("which", range(9))
def test_bad_pointers_bwd(fa, which):
    for bad in (0, P16 + 2):
        ptrs = [P16] * 9
        ptrs[which] = bad
        assert bwd(fa, ptrs=tuple(ptrs)) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_any_finite_scale_passes_the_argument_check(fa):
    # zero and negative scales are valid: the call gets past the checks to the device look-up
    for sc in (0.0, -0.0, -1.0, -1e30, 1e-30):
        assert fwd(fa, scale=sc) == 6
        assert bwd(fa, scale=sc) == 6


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_no_device_fails_loudly(fa):
    # valid arguments without a usable device: an error, never a silent fallback
    assert fwd(fa) == 6
    assert bwd(fa) == 6
    assert fwd8(fa) == 6
    assert step_host(fa) == 6
    with pytest.raises((RuntimeError, ValueError)):
        fa.forward(torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16), torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16),
                   torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16))


def test_debug_set_validates(fa):
    assert fa.fa_debug_set(0, 2) == 1
    assert fa.fa_debug_set(0, 0) == 0


def test_tune_validates(fa):
    # the exp2 split takes 0, 1, 2, 4 or 8; anything else, or an unknown knob, is rejected on the host
    for v in (0, 1, 2, 4, 8):
        assert fa.fa_tune(fa.TUNE_EXP2_SPLIT, v) == 0
    for v in (-1, 3, 16):
        assert fa.fa_tune(fa.TUNE_EXP2_SPLIT, v) == 1
    assert fa.fa_tune(99, 0) == 1
    assert fa.fa_tune(fa.TUNE_EXP2_SPLIT, 0) == 0
    # CTA pairs: 0 or 1
    for v in (-1, 2):
        assert fa.fa_tune(fa.TUNE_CTA_PAIRS, v) == 1
    assert fa.fa_tune(fa.TUNE_CTA_PAIRS, 1) == 0
    assert fa.fa_tune(fa.TUNE_CTA_PAIRS, 0) == 0
    assert fa.fa_tune(fa.TUNE_BWD_SPLIT, -2) == 1
    for v in (5, 0, -1):
        assert fa.fa_tune(fa.TUNE_BWD_SPLIT, v) == 0


def test_bwd_launches_counts(fa):
    # pre-pass, main kernel, dQ conversion; the GQA tail's last pass only when
    # the causal GQA split at d = 128 makes pieces (forced here: one pair per kv head)
    assert fa.fa_bwd_launches(1, 4, 4, 1000, 1000, 128, 1) == 3  # MHA
    assert fa.fa_bwd_launches(2, 8, 2, 1000, 1000, 128, 0) == 3
    assert fa.fa_bwd_launches(2, 8, 2, 1000, 1000, 64, 1) == 3
    assert fa.fa_tune(fa.TUNE_BWD_SPLIT, 1) == 0
    try:
        assert fa.fa_bwd_launches(2, 8, 2, 1000, 1000, 128, 1) == 4
        assert fa.fa_bwd_launches(2, 8, 8, 1000, 1000, 128, 1) == 3  # MHA: no pieces
    finally:
        fa.fa_tune(fa.TUNE_BWD_SPLIT, -1)
    assert fa.fa_bwd_launches(1, 3, 2, 64, 64, 128, 1) == -1  # Hq not a multiple of Hkv
    assert fa.fa_bwd_launches(1, 2, 2, 64, 64, 96, 1) < 0     # unsupported head dim
