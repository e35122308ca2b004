"""Failure handling through the C ABI: injected allocation and launch failures, and
NaN-poisoned empty slots.

Failures are made on the host (ll_debug_inject_fault, LL_FAULT): the library
skips the failing CUDA call and reports it as failed; no device fault is
involved.  An allocation failure in ll_cache_create must return LL_ERR_OOM or
LL_ERR_CUDA, hand back no cache and leave no device memory behind; a launch
failure in a call must return LL_ERR_CUDA and leave the cache's state and slot
bytes as they were, after which the cache keeps matching the float64 oracle.
"""

import os
import subprocess
import sys

import pytest
import torch

import llsynth
from tests.gpu_util import Lockstep

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    torch.cuda.set_device(0)
    return mod


@pytest.mark.parametrize("dtype", ["bf16", "k8", "fp8", "fp32", "fp32-d64"])
def test_allocation_failures_leave_nothing_behind(ll, dtype):
    code = {"bf16": ll.LL_BF16, "k8": ll.LL_BF16_K8, "fp8": ll.LL_FP8, "fp32": ll.LL_FP32,
            "fp32-d64": ll.LL_FP32}[dtype]
    shape = (2, 4, 64 if dtype == "fp32-d64" else 128, 64, 3, 6, 3)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    failures = 0
    for n in range(1, 8):
        ll.ll_debug_inject_fault(ll.LL_FAULT_ALLOC, n)
        try:
            cache = ll.ll_cache_create(*shape, code)
        except ll.LLError as e:
            assert e.status in (ll.LL_ERR_OOM, ll.LL_ERR_CUDA), e
            failures += 1
            torch.cuda.synchronize()
            assert torch.cuda.mem_get_info()[0] == free0, "allocation %d failed but memory was kept" % n
            continue
        # the n-th allocation is past the last one ll_cache_create makes
        ll.ll_debug_inject_fault(ll.LL_FAULT_ALLOC, 0)
        cache.close()
        break
    # bf16: K, V, split scratch, mapped error word; the e4m3 caches add the rounding staging;
    # fp32 at head_dim 128 (CUDA-core kernel) has no scratch, at head_dim 64 (tensor cores) it has
    assert failures == {"bf16": 4, "k8": 5, "fp8": 5, "fp32": 3, "fp32-d64": 4}[dtype]
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_allocation_failure_from_the_environment(ll):
    prog = ("import sys; sys.path.insert(0, %r); import torch; torch.cuda.set_device(0); "
            "import windowed_sink_attention_ll_b300 as ll\n"
            "try:\n    ll.ll_cache_create(1, 2, 64, 16, 3, 6, 3, ll.LL_BF16)\n    print('created')\n"
            "except ll.LLError as e:\n    print('status', e.status)\n" % ROOT)
    out = subprocess.run([sys.executable, "-c", prog], env=dict(os.environ, LL_FAULT="alloc:2"), capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "status %d" % ll.LL_ERR_OOM, out.stdout


@pytest.mark.parametrize("key_fp8", ["bf16", "keys", "kv"])
def test_launch_failures_leave_the_cache_as_it_was(ll, key_fp8):
    H, D, T, S, W, C = 2, 128, 48, 3, 6, 3
    st = Lockstep(ll, 1, H, D, T, S, W, C, torch.bfloat16, key_fp8=(key_fp8 == "keys"), value_fp8=(key_fp8 == "kv"))
    L = C * T

    def chunk(tag):
        return tuple(llsynth.seeded_normal(("faults", key_fp8, tag, t), (L, H, D), device="cuda") for t in "qkv")

    for c in range(4):
        st.attend(0, *chunk(c), commit=True, what="before the faults c%d" % c)
    state = ll.ll_cache_state(st.cache, 0)
    raw = ll.ll_cache_read(st.cache, 0)
    out = torch.empty(L, H, D, dtype=torch.bfloat16, device="cuda")
    # 1: the attention launch of a committing pass fails: nothing enqueued, nothing changed
    # 2: the attention runs, its commit copy fails: the cache is not written, the state not moved
    for n in (1, 2):
        ll.ll_debug_inject_fault(ll.LL_FAULT_LAUNCH, n)
        with pytest.raises(ll.LLError) as e:
            ll.ll_attend_chunk(st.cache, 0, *chunk("fail%d" % n), out, True)
        assert e.value.status == ll.LL_ERR_CUDA
        assert ll.ll_cache_state(st.cache, 0) == state
        k, v = ll.ll_cache_read(st.cache, 0)
        assert torch.equal(k, raw[0]) and torch.equal(v, raw[1])
    # a recache whose copy fails (its prefill attention runs first) changes nothing either
    R = len(st.orc.recache_frames(0))
    win = tuple(llsynth.seeded_normal(("faults-rc", key_fp8, t), (R * T, H, D), device="cuda") for t in "qkv")
    ll.ll_debug_inject_fault(ll.LL_FAULT_LAUNCH, 2)
    with pytest.raises(ll.LLError) as e:
        ll.ll_recache_attend(st.cache, 0, *win, torch.empty_like(win[0]))
    assert e.value.status == ll.LL_ERR_CUDA
    assert ll.ll_cache_state(st.cache, 0) == state
    k, v = ll.ll_cache_read(st.cache, 0)
    assert torch.equal(k, raw[0]) and torch.equal(v, raw[1])
    ll.ll_debug_inject_fault(ll.LL_FAULT_LAUNCH, 0)
    # the cache carries on as if the failed calls had not been made
    for c in range(4, 7):
        st.attend(0, *chunk(c), commit=True, what="after the faults c%d" % c)
        st.check_state()
    st.check_raw(0)
    st.recache_attend(0, *win, what="prefill after the faults")
    st.check_raw(0)
    st.close()


def test_poisoned_empty_slots(ll):
    """Empty slots hold NaN bytes under ll_debug_poison (and again after a reset); outputs stay
    finite and match the oracle, so no attention read a slot without a resident frame."""
    H, D, T, S, W, C = 2, 64, 32, 3, 6, 3
    st = Lockstep(ll, 1, H, D, T, S, W, C, torch.bfloat16)  # poisoned by Lockstep
    L = C * T
    for c in range(2):
        q, k, v = (llsynth.seeded_normal(("poison", c, t), (L, H, D), device="cuda") for t in "qkv")
        st.attend(0, q, k, v, commit=True, what="poisoned c%d" % c)
    hk, hv = ll.ll_cache_read(st.cache, 0)
    n, table = ll.ll_cache_state(st.cache, 0)
    assert n == 6 and table.count(-1) == 3
    for slot, f in enumerate(table):
        empty = f < 0
        assert bool(torch.isnan(hk[:, slot].float()).all()) == empty, slot
        assert bool(torch.isnan(hv[:, slot].float()).all()) == empty, slot
    ll.ll_reset(st.cache)
    st.orc.reset()
    hk, hv = ll.ll_cache_read(st.cache, 0)
    assert bool(torch.isnan(hk.float()).all()) and bool(torch.isnan(hv.float()).all())
    q, k, v = (llsynth.seeded_normal(("poison-after", t), (L, H, D), device="cuda") for t in "qkv")
    st.attend(0, q, k, v, commit=True, what="poisoned after reset")
    st.check_state()
    st.check_raw(0)
    st.close()
