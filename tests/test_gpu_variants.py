"""GPU parity of the two optional readings, through the C ABI, against the oracle:
the frame-causal chunk mask (ll_set_chunk_mask(LL_MASK_FRAME)) and the keep-sink
recache scope (ll_set_recache_scope(LL_RECACHE_WINDOW)).

Same bar as test_gpu_parity.py: attention outputs within max |err| <= 1e-2 and
relative L2 <= 5e-3 of the unrounded float64 oracle; frames committed, the
frame-to-slot map and the raw slot bytes bit-exact after every call.
"""

import numpy as np
import pytest
import torch

import llsynth
import oracle
from tests.gpu_util import Lockstep, sample_rows

pytestmark = pytest.mark.gpu

OPTIONS = [("frame", "resident"), ("chunk", "window"), ("frame", "window")]


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    torch.cuda.set_device(0)
    return mod


def run_small(ll, shape, dtype, mask, scope, chunks=6, tag="var"):
    H, D, T, S, W, C = shape
    st = Lockstep(ll, 2, H, D, T, S, W, C, dtype)
    st.set_options(mask, scope)
    L = C * T
    for c in range(chunks):
        for layer in (0, 1):
            q, k, v = (llsynth.seeded_normal((tag, shape, layer, c, t), (L, H, D), dtype=dtype, device="cuda")
                       for t in "qkv")
            st.attend(layer, q, k, v, commit=True, what="%s %s/%s L%d c%d" % (shape, mask, scope, layer, c))
        st.check_state()
        st.check_raw(0)
        st.check_raw(1)
    R = len(st.orc.recache_frames(1))
    if R:
        qw, kw, vw = (llsynth.seeded_normal((tag + "-rc", shape, t), (R * T, H, D), dtype=dtype, device="cuda")
                      for t in "qkv")
        st.recache_attend(1, qw, kw, vw, what="prefill %s %s/%s" % (shape, mask, scope))
        st.check_state()
        st.check_raw(1)
        kw2, vw2 = (llsynth.seeded_normal((tag + "-rc2", shape, t), (R * T, H, D), dtype=dtype, device="cuda")
                    for t in "kv")
        st.recache(0, kw2, vw2)
        st.check_raw(0)
        q, k, v = (llsynth.seeded_normal((tag + "-after", shape, t), (L, H, D), dtype=dtype, device="cuda")
                   for t in "qkv")
        st.attend(1, q, k, v, commit=False, what="after prefill %s %s/%s" % (shape, mask, scope))
        st.attend(0, q, k, v, commit=False, what="after recache %s %s/%s" % (shape, mask, scope))
    st.close()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("mask,scope", OPTIONS, ids=["%s-%s" % o for o in OPTIONS])
def test_tiny_workload_options(ll, dtype, mask, scope):
    s = llsynth.TINY
    st = Lockstep(ll, s.layers, s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames,
                  s.chunk_frames, dtype)
    st.set_options(mask, scope)
    n_before = llsynth.TINY_RECACHE_BEFORE_CHUNK * s.chunk_frames
    R = None
    inp = llsynth.tiny_inputs(dtype, recache_frames=9)
    for c in range(llsynth.TINY_CHUNKS):
        if c == llsynth.TINY_RECACHE_BEFORE_CHUNK:
            assert st.orc.state(0)[0] == n_before
            R = len(st.orc.recache_frames(0))
            k_win, v_win = (t[-R * s.tokens_per_frame:].cuda() for t in inp["recache_kv"])
            q_win = inp["recache_q"][-R * s.tokens_per_frame:].cuda()
            st.recache_attend(0, q_win, k_win.contiguous(), v_win.contiguous(), what="tiny prefill %s/%s" % (mask, scope))
            st.check_state()
            st.check_raw(0)
        for p in range(llsynth.TINY_PASSES):
            q, k, v = (t.cuda() for t in inp["passes"][c][p])
            st.attend(0, q, k, v, commit=(p == llsynth.TINY_PASSES - 1), what="tiny %s/%s c%d p%d" % (mask, scope, c, p))
            st.check_state()
        st.check_raw(0)
    assert R == (9 if scope == "resident" else 6)
    st.close()


EDGE = [
    # H, d,   T,   S, W, C
    (2, 64, 8, 4, 2, 3),       # window shorter than a chunk, sink longer than a chunk
    (3, 128, 24, 2, 4, 3),     # sink shorter than a chunk
    (2, 128, 100, 3, 9, 3),    # 300 queries (2 query tiles, ragged), frame blocks of 100 keys
    (1, 128, 200, 3, 3, 2),    # 400 queries: 2 CTAs per head, ragged second one
    (2, 64, 37, 0, 6, 3),      # no sink, odd T
    (2, 64, 5, 2, 4, 1),       # one-frame chunks: the frame mask is the chunk mask
]


@pytest.mark.parametrize("shape", EDGE, ids=["-".join(map(str, e)) for e in EDGE])
@pytest.mark.parametrize("mask,scope", OPTIONS, ids=["%s-%s" % o for o in OPTIONS])
def test_edge_shapes_options(ll, shape, mask, scope):
    run_small(ll, shape, torch.bfloat16, mask, scope)


def test_edge_fp32_frame_mask(ll):
    run_small(ll, (2, 64, 37, 3, 6, 3), torch.float32, "frame", "window")


def wan(tag, layer, c, shape, per_head=False):
    L = shape.chunk_tokens
    return tuple(llsynth.seeded_normal((tag, layer, c, t), (L, shape.heads, shape.head_dim), device="cuda",
                                       per_head_scale=per_head) for t in "qkv")


def test_single_layer_wan_frame_mask(ll):
    """Wan-shaped layer at steady state with the frame-causal chunk: 228 work items on the
    SMs, left-over items split and merged; fp32 output so the kernel's own error is held
    to 1e-2 (per-head scales up to 2 make |o| reach 4)."""
    s = llsynth.SINGLE_LAYER
    st = Lockstep(ll, 1, s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames,
                  s.chunk_frames, torch.bfloat16)
    st.set_options("frame", "resident")
    ll.ll_set_output_dtype(st.cache, torch.float32)
    for c in range(4):
        st.attend(0, *wan("var-single", 0, c, s, per_head=True), commit=True, check=False)
    rows = sample_rows(s.chunk_tokens, 512)
    # rows of all three frames of the chunk, including the frame boundaries
    T = s.tokens_per_frame
    rows = np.unique(np.concatenate([rows, [T - 1, T, 2 * T - 1, 2 * T]]))
    for p in range(2):
        st.attend(0, *wan("var-single-pass%d" % p, 0, 4, s, per_head=True), commit=(p == 1), rows=rows,
                  what="single layer frame mask pass %d" % p)
        st.check_state()
    st.check_raw(0)
    st.close()


def test_wan_keep_sink_recache_prefill(ll):
    """The prompt-switch prefill with the keep-sink scope at Wan shapes: 9 window frames
    (14040 queries) attend to the 3 cached sink frames plus the fresh window."""
    s = llsynth.RECACHE30
    st = Lockstep(ll, 1, s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames,
                  s.chunk_frames, torch.bfloat16, keep_frames=False)
    st.set_options("chunk", "window")
    for c in range(10):
        st.attend(0, *wan("var-rc", 0, c, s), commit=True, check=False)
    frames = st.orc.recache_frames(0)
    assert frames == list(range(21, 30))
    L = len(frames) * s.tokens_per_frame
    qw, kw, vw = (llsynth.seeded_normal(("var-rc-win", t), (L, s.heads, s.head_dim), device="cuda") for t in "qkv")
    st.recache_attend(0, qw, kw, vw, rows=sample_rows(L, 384, seed=3), what="keep-sink prefill")
    st.check_state()
    st.attend(0, *wan("var-rc-after", 0, 10, s), commit=True, rows=sample_rows(s.chunk_tokens, 256),
              what="attend after keep-sink prefill")
    st.close()


def test_window_scope_without_window_frames_is_a_state_error(ll):
    st = Lockstep(ll, 1, 2, 64, 16, 3, 6, 3, torch.bfloat16)
    st.set_options("chunk", "window")
    q, k, v = (llsynth.seeded_normal(("var-state", t), (48, 2, 64), device="cuda") for t in "qkv")
    st.attend(0, q, k, v, commit=True)  # only the sink is resident now
    with pytest.raises(ll.LLError) as e:
        ll.ll_recache(st.cache, 0, k, v)
    assert e.value.status == ll.LL_ERR_STATE
    st.close()


def test_option_setters_reject_unknown_values(ll):
    cache = ll.ll_cache_create(1, 2, 64, 16, 3, 6, 3, ll.LL_BF16)
    for setter in (ll.ll_set_chunk_mask, ll.ll_set_recache_scope):
        for bad in (-1, 2, 7):
            with pytest.raises(ll.LLError) as e:
                setter(cache, bad)
            assert e.value.status == ll.LL_ERR_INVALID_ARG
    ll.ll_set_chunk_mask(cache, "frame")
    ll.ll_set_recache_scope(cache, "window")
    cache.close()
