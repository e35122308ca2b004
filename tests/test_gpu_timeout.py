"""Bounded device waits: a wait that runs out reports an error and leaves the context usable.

ll_debug_inject_stall makes the next tensor-core attention launch skip the first
P-ready arrival of query tile 0, so the MMA thread's wait for it can never be
satisfied (a barrier phase that nothing completes).  The wait gives up after the
given limit, the CTA leaves its loops, drains its copies and MMAs and frees its
tensor memory; the next ll_sync reports LL_ERR_DEVICE_TIMEOUT once, and later
calls run normally and match the oracle.  No trap, assert or bad address is used.
"""

import pytest
import torch

import llsynth
from tests.gpu_util import Lockstep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    torch.cuda.set_device(0)
    return mod


@pytest.mark.parametrize("T,pair,kind", [(16, False, "bf16"), (1040, False, "bf16"), (1040, True, "bf16"),
                                         (16, False, "fp32"), (1040, False, "fp32"), (1040, False, "fp8")],
                         ids=["one-cta-small", "one-cta-persistent", "cta-pair-persistent", "tf32-small",
                              "tf32-persistent", "fp8-persistent"])
def test_stalled_wait_times_out_and_the_cache_keeps_working(ll, T, pair, kind):
    """T = 16: one CTA per head pair; T = 1040: a persistent grid with split items, on the
    one-CTA kernel and on the CTA-pair kernel (whose two CTAs must both give up and meet
    before they free tensor memory), on the one-CTA kernel with fp32 operands (tf32,
    head_dim 64), whose K-split / V-transpose warps wait as well, and with e4m3 keys and
    values, whose V-widening warps wait."""
    fp32 = kind == "fp32"
    H, D, S, W, C = (2, 64, 3, 6, 3) if T == 16 else (12, 64 if fp32 else 128, 3, 6, 3)
    dtype = torch.float32 if fp32 else torch.bfloat16
    st = Lockstep(ll, 1, H, D, T, S, W, C, dtype, value_fp8=(kind == "fp8"))
    ll.ll_debug_pair_kernel(st.cache, pair)
    L = C * T
    for c in range(3):
        q, k, v = (llsynth.seeded_normal(("stall", T, c, t), (L, H, D), dtype=dtype, device="cuda") for t in "qkv")
        st.attend(0, q, k, v, commit=True, what="before the stall c%d" % c)
    state = ll.ll_cache_state(st.cache, 0)
    q, k, v = (llsynth.seeded_normal(("stall-q", T, pair, t), (L, H, D), dtype=dtype, device="cuda")
               for t in "qkv")
    ll.ll_debug_inject_stall(st.cache, True, 20000)  # 20 ms limit for the next launch's waits
    out = torch.empty_like(q)
    ll.ll_attend_chunk(st.cache, 0, q, k, v, out, False)  # enqueued fine; the device wait gives up
    with pytest.raises(ll.LLError) as e:
        ll.ll_sync(st.cache)
    assert e.value.status == ll.LL_ERR_DEVICE_TIMEOUT
    ll.ll_sync(st.cache)  # reported once
    assert ll.ll_cache_state(st.cache, 0) == state
    # the context and the cache still work: the same pass again, then commits, against the oracle
    st.attend(0, q, k, v, commit=False, what="after the stall")
    for c in range(3, 5):
        q, k, v = (llsynth.seeded_normal(("stall", T, c, t), (L, H, D), dtype=dtype, device="cuda") for t in "qkv")
        st.attend(0, q, k, v, commit=True, what="after the stall c%d" % c)
    st.check_state()
    st.check_raw(0)
    st.close()
