"""fp32 attention on the tensor cores (tf32 operands), head_dim 64, against the oracle.

A cache of dtype fp32 at head_dim 64 runs the one-CTA tensor-core kernel with
kind::tf32 MMAs: Q K^T reads q and k as tf32, P is rounded to tf32 before P V,
and V is transposed in shared memory into the K-major layout P V reads.  What it
computes is the attention of "LongLive", §3.3 "Frame sink" + "Short window
attention" (chunk attend) and §3.1 "KV recache" (block-causal prefill); the
outputs must match the float64 oracle within max |err| <= 1e-2 and relative L2
<= 5e-3 through ragged tiles, several key tiles, split tails (many heads), both
chunk masks and both recache scopes, with cache state and slot bytes bit-exact.
The CUDA-core kernel (ll_debug_use_simt) gives a second opinion on the same
passes.
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
    (1, 5, 0, 0, 1),      # 5 queries, 5 keys: one tile, mostly padding
    (2, 16, 3, 6, 3),     # the tiny workload's shape
    (3, 100, 3, 9, 3),    # 300 queries (2 items per head, ragged), up to 1500 keys
    (2, 130, 2, 3, 2),    # tiles that straddle the cache / chunk boundary
    (64, 200, 2, 4, 3),   # 192 items: a whole round of CTAs, then a split tail merged in fp32
]


@pytest.mark.parametrize("scope", ["resident", "window"])
@pytest.mark.parametrize("mask", ["chunk", "frame"])
@pytest.mark.parametrize("shape", SHAPES, ids=["-".join(map(str, s)) for s in SHAPES])
def test_fp32_tensor_core_path(ll, shape, mask, scope):
    H, T, S, W, C = shape
    D = 64
    st = Lockstep(ll, 1, H, D, T, S, W, C, torch.float32)
    st.set_options(chunk_mask=mask, recache_scope=scope)
    L = C * T
    for c in range(5):
        q, k, v = (llsynth.seeded_normal(("tf32", shape, mask, c, t), (L, H, D), dtype=torch.float32,
                                         device="cuda") for t in "qkv")
        st.attend(0, q, k, v, commit=True, what="tf32 %s %s chunk %d" % (shape, mask, c))
        st.check_state()
    st.check_raw(0)
    R = len(st.orc.recache_frames(0))
    if R:  # nothing to rewrite without a sink or a window (or, keeping the sink, without a window)
        qw, kw, vw = (llsynth.seeded_normal(("tf32-rc", shape, mask, t), (R * T, H, D), dtype=torch.float32,
                                            device="cuda") for t in "qkv")
        st.recache_attend(0, qw, kw, vw, what="tf32 prefill %s %s %s" % (shape, mask, scope))
        st.check_state()
        st.check_raw(0)
    q, k, v = (llsynth.seeded_normal(("tf32-after", shape, mask, t), (L, H, D), dtype=torch.float32, device="cuda")
               for t in "qkv")
    st.attend(0, q, k, v, commit=False, what="tf32 after prefill %s %s" % (shape, mask))
    st.close()


def test_fp32_tensor_core_and_cuda_core_kernels_agree(ll):
    """The tf32 tensor-core kernel and the fp32 CUDA-core kernel on the same passes, each
    within the bound of the oracle (Lockstep checks every output), and within 2e-2 of
    each other."""
    H, D, T, S, W, C = 3, 64, 70, 3, 6, 3
    outs = []
    for simt in (False, True):
        st = Lockstep(ll, 1, H, D, T, S, W, C, torch.float32)
        ll.ll_debug_use_simt(st.cache, simt)
        for c in range(4):
            q, k, v = (llsynth.seeded_normal(("tf32-agree", c, t), (C * T, H, D), dtype=torch.float32,
                                             device="cuda") for t in "qkv")
            outs.append(st.attend(0, q, k, v, commit=True, what="fp32 simt=%s c%d" % (simt, c)))
        st.close()
    for a, b in zip(outs[:4], outs[4:]):
        assert float((a.double() - b.double()).abs().max()) <= 2e-2


def test_fp32_large_scores_split_tail(ll):
    """Per-head scales 0.5-2 (scores up to ~4x those of unit inputs) on a persistent grid
    with split items: the tf32 operands' 10-bit mantissas still keep the outputs within
    the bound (sampled rows of the last pass)."""
    H, D, T, S, W, C = 24, 64, 520, 3, 9, 3
    st = Lockstep(ll, 1, H, D, T, S, W, C, torch.float32, keep_frames=False)
    L = C * T
    for c in range(5):
        q, k, v = (llsynth.seeded_normal(("tf32-scaled", c, t), (L, H, D), dtype=torch.float32, device="cuda",
                                         per_head_scale=True) for t in "qkv")
        last = c == 4
        st.attend(0, q, k, v, commit=True, check=last, rows=sample_rows(L, 256, seed=5) if last else None,
                  what="tf32 scaled chunk %d" % c)
    st.check_state()
    st.close()
