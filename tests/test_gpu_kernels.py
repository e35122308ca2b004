"""The two tensor-core attention kernels at head_dim 128, each against the oracle.

head_dim 128 runs on the one-CTA kernel by default (the kernel every bf16
attention uses); ll_debug_pair_kernel routes a cache to the CTA-pair kernel (two
SMs share every MMA, M = 256).  Both must match the float64 oracle ("LongLive", §3.3 "Frame sink" +
"Short window attention" for the chunk attend, §3.1 "KV recache" for the
prefill) within max |err| <= 1e-2 and relative L2 <= 5e-3, on the chunk-mask and
frame-mask attends and on the block-causal prefill, through ragged tiles, a
split tail and a persistent prefill grid; cache state and slot bytes bit-exact.
"""

import pytest
import torch

import llsynth
from tests.gpu_util import Lockstep, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    torch.cuda.set_device(0)
    return mod


SHAPES = [
    # H,  T,   S, W, C
    (1, 5, 0, 0, 1),      # 5 queries: one pair, the second CTA's rows all past the end
    (3, 100, 3, 9, 3),    # 300 queries (2 items per head, ragged), up to 1500 keys: partial K halves
    (2, 130, 2, 3, 2),    # tiles that straddle the cache / chunk boundary
    (64, 200, 2, 4, 3),   # 192 items: a whole round of pairs, then a split tail
]


@pytest.mark.parametrize("pair", [True, False], ids=["pair", "one_cta"])
@pytest.mark.parametrize("mask", ["chunk", "frame"])
@pytest.mark.parametrize("shape", SHAPES, ids=["-".join(map(str, s)) for s in SHAPES])
def test_head_dim_128_kernels(ll, shape, mask, pair):
    H, T, S, W, C = shape
    D = 128
    st = Lockstep(ll, 1, H, D, T, S, W, C, torch.bfloat16)
    ll.ll_debug_pair_kernel(st.cache, pair)
    st.set_options(chunk_mask=mask)
    L = C * T
    for c in range(5):
        q, k, v = (llsynth.seeded_normal(("kernels", shape, mask, c, t), (L, H, D), device="cuda") for t in "qkv")
        st.attend(0, q, k, v, commit=True, what="%s %s %s chunk %d" % ("pair" if pair else "one_cta", shape,
                                                                         mask, c))
        st.check_state()
    st.check_raw(0)
    R = len(st.orc.recache_frames(0))
    if R:  # nothing is resident without a sink or a window
        qw, kw, vw = (llsynth.seeded_normal(("kernels-rc", shape, mask, t), (R * T, H, D), device="cuda")
                      for t in "qkv")
        st.recache_attend(0, qw, kw, vw, what="%s prefill %s %s" % ("pair" if pair else "one_cta", shape, mask))
        st.check_state()
        st.check_raw(0)
    q, k, v = (llsynth.seeded_normal(("kernels-after", shape, mask, t), (L, H, D), device="cuda") for t in "qkv")
    st.attend(0, q, k, v, commit=False, what="after prefill %s %s" % (shape, mask))
    st.close()


def test_wan_layer_both_kernels_fp32_out(ll):
    """The single Wan-shaped layer (per-head scales 0.5-2, 23400 keys) with fp32 outputs on
    both kernels: each within the strict bound of the oracle on sampled rows."""
    s = llsynth.SINGLE_LAYER
    rows = sample_rows(s.chunk_tokens, 256, seed=11)
    for pair in (True, False):
        st = Lockstep(ll, 1, s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames,
                      s.chunk_frames, torch.bfloat16, keep_frames=False)
        ll.ll_debug_pair_kernel(st.cache, pair)
        ll.ll_set_output_dtype(st.cache, torch.float32)
        for c in range(4):
            q, k, v = (llsynth.seeded_normal(("kernels-wan", c, t), (s.chunk_tokens, s.heads, s.head_dim),
                                             device="cuda", per_head_scale=True) for t in "qkv")
            st.attend(0, q, k, v, commit=True, check=False)
        q, k, v = (llsynth.seeded_normal(("kernels-wan-q", t), (s.chunk_tokens, s.heads, s.head_dim), device="cuda",
                                         per_head_scale=True) for t in "qkv")
        st.attend(0, q, k, v, commit=True, rows=rows, what="Wan layer fp32 out, %s" % ("pair" if pair
                                                                                        else "one_cta"))
        st.check_state()
        st.close()
