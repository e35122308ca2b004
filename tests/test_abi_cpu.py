"""CPU-only checks of the C-ABI library: it builds, loads, exports every symbol the
header declares, and its host-side index logic matches the oracle bit for bit."""

import os
import re

import pytest
import torch

import oracle
from tests.conftest import ROOT


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    return mod


def header_symbols():
    text = open(os.path.join(ROOT, "include", "ll.h")).read()
    return sorted(set(re.findall(r"^LL_API [^(]*?\b(ll_\w+)\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol(ll):
    declared = header_symbols()
    assert len(declared) >= 16
    lib = ll._lib()
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(ll.EXPORTS) == declared


def test_binding_names_match_the_abi(ll):
    for name in header_symbols():
        assert callable(getattr(ll, name)), name


def test_frame_slot_matches_oracle(ll):
    for S in range(0, 6):
        for W in range(0, 8):
            for f in range(0, 60):
                want = oracle.slot_of_frame(S, W, f) if (f < S or W > 0) else -1
                assert ll.ll_frame_slot(S, W, f) == want


def test_resident_frames_match_oracle(ll):
    for S in range(0, 6):
        for W in range(0, 8):
            for n in range(0, 80):
                assert ll.ll_resident_frames(S, W, n) == oracle.resident_frames(S, W, n)


def test_resident_slots_form_a_prefix(ll):
    # the kernels read resident keys as slots [0, R): check that claim for many shapes
    for S in range(0, 6):
        for W in range(0, 8):
            for C in range(1, 5):
                for n in range(0, 60, C):
                    frames = ll.ll_resident_frames(S, W, n)
                    slots = sorted(ll.ll_frame_slot(S, W, f) for f in frames)
                    assert slots == list(range(len(frames)))


def test_status_strings(ll):
    assert [ll.ll_status_str(i) for i in range(7)] == ll.STATUS


def test_create_rejects_bad_arguments_before_touching_a_device(ll):
    bad = [
        (0, 2, 64, 16, 3, 6, 3, ll.LL_BF16),
        (1, 0, 64, 16, 3, 6, 3, ll.LL_BF16),
        (1, 2, 64, 0, 3, 6, 3, ll.LL_BF16),
        (1, 2, 64, 16, -1, 6, 3, ll.LL_BF16),
        (1, 2, 64, 16, 3, -1, 3, ll.LL_BF16),
        (1, 2, 64, 16, 3, 6, 0, ll.LL_BF16),
        (1, 2, 64, 16, 3, 6, 3, 7),
    ]
    for args in bad:
        with pytest.raises(ll.LLError) as e:
            ll.ll_cache_create(*args)
        assert e.value.status == ll.LL_ERR_INVALID_ARG, args
    too_big = [
        (1, 2, 96, 16, 3, 6, 3, ll.LL_BF16),         # head_dim not 64 / 128
        (1, 2, 64, 16, 400, 200, 3, ll.LL_BF16),     # S + W = 600 > 512 frames
        (1, 2, 64, 16, 3, 6, 513, ll.LL_BF16),       # C = 513 > 512 frames
        (1, 128, 64, 16, 3, 6, 3, ll.LL_BF16),       # 128 heads > 127
        (1, 2, 64, 1 << 27, 3, 6, 3, ll.LL_BF16),    # (S + W + C) * T = 12 * 2^27 > 2^30 tokens
    ]
    for args in too_big:
        with pytest.raises(ll.LLError) as e:
            ll.ll_cache_create(*args)
        assert e.value.status == ll.LL_ERR_UNSUPPORTED, args


@pytest.mark.skipif(torch.cuda.is_available(), reason="at the limits a GPU would allocate")
def test_create_limits_are_inclusive(ll):
    # exactly at each limit the request passes every size check and stops at the
    # device lookup (no GPU here)
    at_limit = [
        (1, 2, 64, 16, 500, 12, 3, ll.LL_BF16),      # S + W = 512
        (1, 2, 64, 16, 3, 6, 512, ll.LL_BF16),       # C = 512
        (1, 127, 64, 16, 3, 6, 3, ll.LL_BF16),       # 127 heads
        (1, 2, 64, 1 << 26, 8, 5, 3, ll.LL_BF16),    # (S + W + C) * T = 16 * 2^26 = 2^30
    ]
    for args in at_limit:
        with pytest.raises(ll.LLError) as e:
            ll.ll_cache_create(*args)
        assert e.value.status == ll.LL_ERR_CUDA, args


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_create_without_a_device_fails_cleanly(ll):
    with pytest.raises(ll.LLError) as e:
        ll.ll_cache_create(1, 2, 64, 16, 3, 6, 3, ll.LL_BF16)
    assert e.value.status == ll.LL_ERR_CUDA


def test_null_handle_calls_return_invalid_arg(ll):
    lib = ll._lib()
    assert lib.ll_reset(None) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_sync(None) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_attend_chunk(None, 0, None, None, None, None, 0, None) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_recache(None, 0, None, None, None) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_recache_attend(None, 0, None, None, None, None, None) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_cache_state(None, 0, None, None) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_cache_read(None, 0, None, None) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_cache_info(None, None, None, None) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_debug_inject_stall(None, 1, 10) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_recache_tokens(None, 0, None) == ll.LL_ERR_INVALID_ARG
    lib.ll_cache_destroy(None)


def test_binding_rejects_host_tensors(ll):
    cache = ll.LLCache(None, 1, 2, 64, 16, 3, 6, 3, ll.LL_BF16)
    t = torch.zeros(48, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ll.ll_attend_chunk(cache, 0, t, t, t, t, True)


def test_noalloc_rejects_an_output_that_overlaps_an_input(ll):
    """Byte-range checks of ll_attend_chunk_noalloc.  They run before the call looks
    at a device: every overlapping case returns LL_ERR_INVALID_ARG, and each
    control without the overlap stops at the head_dim check (96: LL_ERR_UNSUPPORTED).
    The addresses are never dereferenced and nothing is enqueued."""
    lib = ll._lib()
    L, H, d = 64, 2, 96
    nb = L * H * d * 2  # bytes of q, k, v and out
    base = 1 << 40
    q, k, v = base, base + (1 << 20), base + (2 << 20)
    kc, vc = base + (8 << 20), base + (12 << 20)
    cached, stride = 100, 100 * d
    cb = ((H - 1) * stride + cached * d) * 2  # bytes spanned by the cached rows of all heads

    def call(out, cached_tokens=cached):
        return lib.ll_attend_chunk_noalloc(q, kc, vc, cached_tokens, stride, k, v, L, out, H, d, None, None)

    for out in (q, q + 16, q - nb + 16, k + nb - 16, v - nb + 16, kc + cb - 16, vc - nb + 16):
        assert call(out) == ll.LL_ERR_INVALID_ARG, hex(out - base)
    for out in (base + (4 << 20), q + nb, q - nb, kc + cb, vc - nb):
        assert call(out) == ll.LL_ERR_UNSUPPORTED, hex(out - base)
    # with no cached rows the cached pointers are ignored
    assert call(kc, cached_tokens=0) == ll.LL_ERR_UNSUPPORTED


def test_e4m3_rounding_helper_matches_the_format_definition():
    """The tests' e4m3 rounding (torch conversion after a clamp to +-448) against rounding
    written from the format: 3 mantissa bits, exponent bias 7 (normals down to 2^-6, then
    subnormals spaced 2^-9), nearest value with ties to even, saturating at +-448."""
    import numpy as np
    import torch

    from tests.gpu_util import round_e4m3

    def e4m3_from_definition(x):
        ax = np.abs(x)
        e = np.maximum(np.floor(np.log2(np.maximum(ax, 2.0 ** -30))), -6)
        step = 2.0 ** (e - 3)
        return np.sign(x) * np.minimum(np.round(ax / step) * step, 448.0)

    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(20000) * s for s in (0.003, 0.05, 1, 8, 100)]
    ties = [(8 + m) * 2.0 ** (e - 3) + 2.0 ** (e - 4) for e in range(-6, 9) for m in range(8)]
    ties += [m * 2.0 ** -9 + 2.0 ** -10 for m in range(8)]
    vals += [np.array(ties), -np.array(ties), np.array([447.9, 448.0, 460.0, 470.0, 1000.0, -1000.0, 0.0])]
    x = torch.from_numpy(np.concatenate(vals)).to(torch.bfloat16)
    got = round_e4m3(x).double().numpy()
    want = e4m3_from_definition(x.double().numpy())
    assert np.array_equal(got, want)


def test_fault_injection_arguments():
    """ll_debug_inject_fault takes a known kind and n >= 0 (host only)."""
    import windowed_sink_attention_ll_b300 as ll

    lib = ll._lib()
    assert lib.ll_debug_inject_fault(ll.LL_FAULT_ALLOC, 0) == ll.LL_OK
    assert lib.ll_debug_inject_fault(ll.LL_FAULT_LAUNCH, 0) == ll.LL_OK
    assert lib.ll_debug_inject_fault(7, 1) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_debug_inject_fault(ll.LL_FAULT_ALLOC, -1) == ll.LL_ERR_INVALID_ARG
    assert lib.ll_debug_poison(None, 1) == ll.LL_ERR_INVALID_ARG
