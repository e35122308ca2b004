"""GPU parity: libll (through its C ABI) against the float64 oracle.

Attention outputs: max |err| <= 1e-2 and relative L2 <= 5e-3 against the
unrounded float64 oracle on the same (dtype-rounded) inputs.  Cache state
(frames committed, frame-to-slot map) and the raw slot bytes: bit-exact.

Chunk numbering: the five workloads are described with 1-based chunk numbers
where the text says "checked at chunks 1, 2, 4, 80 and 320" (chunk 320 is the
last of 320), and with switch points "at chunks 10, 20, 30" read as: the
recache runs after 10 / 20 / 30 chunks were committed, before the attend of
0-based chunk 10 / 20 / 30.
"""

import numpy as np
import pytest
import torch

import llsynth
import oracle
from tests.gpu_util import Lockstep, compare, f64, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    torch.cuda.set_device(0)
    return mod


def dev(t):
    return t.cuda()


# ---------------------------------------------------------------------------
# Tiny workload: every output row, every call
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("prefill", [False, True])
def test_tiny_workload(ll, dtype, prefill):
    s = llsynth.TINY
    st = Lockstep(ll, s.layers, s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames,
                  s.chunk_frames, dtype)
    # resident frames before chunk 5: 3 sink + 6 window
    n_before = llsynth.TINY_RECACHE_BEFORE_CHUNK * s.chunk_frames
    R = len(oracle.resident_frames(s.sink_frames, s.window_frames, n_before))
    assert R == 9
    inp = llsynth.tiny_inputs(dtype, recache_frames=R)
    for c in range(llsynth.TINY_CHUNKS):
        if c == llsynth.TINY_RECACHE_BEFORE_CHUNK:
            k_win, v_win = (dev(t) for t in inp["recache_kv"])
            if prefill:
                st.recache_attend(0, dev(inp["recache_q"]), k_win, v_win, what="tiny prefill")
            else:
                st.recache(0, k_win, v_win)
            st.check_state()
            st.check_raw(0)
        for p in range(llsynth.TINY_PASSES):
            q, k, v = (dev(t) for t in inp["passes"][c][p])
            st.attend(0, q, k, v, commit=(p == llsynth.TINY_PASSES - 1), what="tiny c%d p%d" % (c, p))
            st.check_state()
        st.check_raw(0)
    st.close()


def test_tensor_core_and_cuda_core_kernels_agree(ll):
    """Both CUDA kernels of the bf16 path against the oracle on one pass each."""
    H, D, T, S, W, C = 2, 128, 50, 3, 6, 3
    outs = []
    for simt in (False, True):
        st = Lockstep(ll, 1, H, D, T, S, W, C, torch.bfloat16)
        ll.ll_debug_use_simt(st.cache, simt)
        for c in range(4):
            q, k, v = (llsynth.seeded_normal(("agree", c, t), (C * T, H, D), device="cuda") for t in "qkv")
            outs.append(st.attend(0, q, k, v, commit=True, what="simt=%s c%d" % (simt, c)))
        st.close()
    for a, b in zip(outs[:4], outs[4:]):
        assert float((a.double() - b.double()).abs().max()) <= 2e-2


# ---------------------------------------------------------------------------
# Edge cases: ragged sizes, no sink / no window, W < C, S > C, several tiles
# ---------------------------------------------------------------------------

EDGE = [
    # H, d,   T,   S, W, C
    (1, 64, 5, 0, 0, 1),       # no cache at all: plain attention inside a 5-token chunk
    (2, 64, 8, 4, 2, 3),       # window shorter than a chunk, sink longer than a chunk
    (3, 128, 24, 2, 4, 3),     # sink shorter than a chunk
    (2, 128, 100, 3, 9, 3),    # 300 queries (2 query tiles, ragged), up to 1500 keys
    (1, 128, 200, 3, 3, 2),    # 400 queries: 2 CTAs per head, ragged second one
    (2, 64, 37, 0, 6, 3),      # no sink, odd T
    (2, 128, 33, 3, 0, 3),     # sink only
]


@pytest.mark.parametrize("shape", EDGE, ids=["-".join(map(str, e)) for e in EDGE])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_edge_shapes(ll, shape, dtype):
    H, D, T, S, W, C = shape
    st = Lockstep(ll, 2, H, D, T, S, W, C, dtype)
    L = C * T
    for c in range(6):
        for layer in (0, 1):
            q, k, v = (llsynth.seeded_normal(("edge", shape, layer, c, t), (L, H, D), dtype=dtype, device="cuda")
                       for t in "qkv")
            st.attend(layer, q, k, v, commit=True, what="edge %s L%d c%d" % (shape, layer, c))
        st.check_state()
        st.check_raw(0)
        st.check_raw(1)
    R = len(st.orc.resident(1))
    if R:
        qw, kw, vw = (llsynth.seeded_normal(("edge-rc", shape, t), (R * T, H, D), dtype=dtype, device="cuda")
                      for t in "qkv")
        st.recache_attend(1, qw, kw, vw, what="edge prefill %s" % (shape,))
        st.check_state()
        st.check_raw(1)
        q, k, v = (llsynth.seeded_normal(("edge-after", shape, t), (L, H, D), dtype=dtype, device="cuda")
                   for t in "qkv")
        st.attend(1, q, k, v, commit=False, what="edge after recache %s" % (shape,))
    st.close()


def test_reset_and_empty_recache(ll):
    st = Lockstep(ll, 2, 2, 64, 16, 3, 6, 3, torch.bfloat16)
    z = torch.zeros(144, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ll.LLError) as e:
        ll.ll_recache(st.cache, 0, z, z)
    assert e.value.status == ll.LL_ERR_STATE
    for c in range(3):
        q, k, v = (llsynth.seeded_normal(("reset", c, t), (48, 2, 64), device="cuda") for t in "qkv")
        st.attend(0, q, k, v, commit=True)
    ll.ll_reset(st.cache)
    st.orc.reset()
    st.check_state()
    q, k, v = (llsynth.seeded_normal(("reset-after", t), (48, 2, 64), device="cuda") for t in "qkv")
    st.attend(0, q, k, v, commit=False, what="attend after reset")
    with pytest.raises(ll.LLError) as e:
        ll.ll_attend_chunk(st.cache, 2, q, k, v, torch.empty_like(q), True)
    assert e.value.status == ll.LL_ERR_INVALID_ARG
    st.check_state()
    # a recache window of the wrong length is refused before the library reads it
    assert ll.ll_recache_tokens(st.cache, 0) == 0
    st.attend(0, q, k, v, commit=True, what="commit after reset")
    assert ll.ll_recache_tokens(st.cache, 0) == 3 * 16
    short = torch.zeros(2 * 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        ll.ll_recache(st.cache, 0, short, short)
    st.check_state()
    st.check_raw(0)
    st.close()


def test_output_sharing_bytes_with_an_input_is_rejected(ll):
    """An output that shares any byte with an input (q, k, v; q_win, k_win, v_win) is
    rejected before anything is enqueued, and the cache is left as it was.  All
    tensors are views of one allocation with the inputs at byte offsets 2nb, 3nb,
    4nb (nb = bytes of one bf16 input), so no case reaches outside it."""
    H, D, T, S, W, C = 2, 64, 16, 3, 6, 3
    st = Lockstep(ll, 1, H, D, T, S, W, C, torch.bfloat16)

    def buffer(rows, tag):
        nb = rows * H * D * 2
        raw = torch.zeros(8 * nb, dtype=torch.uint8, device="cuda")

        def at(off, dt=torch.bfloat16):
            size = nb * (2 if dt == torch.float32 else 1)
            return raw[off:off + size].view(dt).view(rows, H, D)

        ins = [at(i * nb) for i in (2, 3, 4)]
        for t, name in zip(ins, "qkv"):
            t.copy_(llsynth.seeded_normal((tag, name), (rows, H, D), device="cuda"))
        return nb, at, ins

    L = C * T
    nb, at, (q, k, v) = buffer(L, "overlap")
    for off in (nb + 16, 2 * nb + 16, 3 * nb - 16, 4 * nb + 16, 5 * nb - 16):
        with pytest.raises(ll.LLError) as e:
            ll.ll_attend_chunk(st.cache, 0, q, k, v, at(off), True)
        assert e.value.status == ll.LL_ERR_INVALID_ARG, off
    # an fp32 output is 2nb long: at byte 16 it ends 16 bytes inside q
    ll.ll_set_output_dtype(st.cache, torch.float32)
    with pytest.raises(ll.LLError) as e:
        ll.ll_attend_chunk(st.cache, 0, q, k, v, at(16, torch.float32), True)
    assert e.value.status == ll.LL_ERR_INVALID_ARG
    st.check_state()
    # outputs that end at q's first byte or start after v's last are accepted
    want = st.orc.attend(0, f64(q), f64(k), f64(v), False)
    out32 = at(0, torch.float32)
    ll.ll_attend_chunk(st.cache, 0, q, k, v, out32, False)
    compare(out32, want, "fp32 out ending where q starts")
    ll.ll_set_output_dtype(st.cache, torch.bfloat16)
    out = at(5 * nb)
    st.orc.attend(0, f64(q), f64(k), f64(v), True)  # same pass, committed on both sides
    ll.ll_attend_chunk(st.cache, 0, q, k, v, out, True)
    compare(out, want, "bf16 out starting after v")
    st.host[0].update({i: (k[i * T:(i + 1) * T].cpu(), v[i * T:(i + 1) * T].cpu()) for i in range(C)})
    q2, k2, v2 = (llsynth.seeded_normal(("overlap-2", t), (L, H, D), device="cuda") for t in "qkv")
    st.attend(0, q2, k2, v2, commit=True)
    st.check_state()
    st.check_raw(0)

    R = 6  # resident frames after two chunks: 3 sink + 3 window
    nbw, atw, (qw, kw, vw) = buffer(R * T, "overlap-rc")
    for off in (nbw + 16, 3 * nbw + 16, 5 * nbw - 16):
        with pytest.raises(ll.LLError) as e:
            ll.ll_recache_attend(st.cache, 0, qw, kw, vw, atw(off))
        assert e.value.status == ll.LL_ERR_INVALID_ARG, off
    st.check_state()
    st.check_raw(0)
    st.close()


# ---------------------------------------------------------------------------
# Wan-shaped workloads at full size (sampled query rows, all heads)
# ---------------------------------------------------------------------------


def wan_chunk(tag, layer, c, shape, per_head=False):
    L = shape.chunk_tokens
    return tuple(llsynth.seeded_normal((tag, layer, c, t), (L, shape.heads, shape.head_dim), device="cuda",
                                       per_head_scale=per_head) for t in "qkv")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_single_layer_wan(ll, out_dtype):
    """Per-head scales up to 2 on q, k and v make |o| reach 4 and more, where rounding the
    output to bf16 alone can cost up to |o| * 2^-9 > 1e-2.  With fp32 output the kernel's
    own error is held to max|err| <= 1e-2 against the unrounded oracle; with bf16 output
    every element must be the bf16 rounding of a value within 1e-2 of the oracle (and at
    most one ulp from bf16(oracle)); relative L2 <= 5e-3 against the unrounded oracle
    either way."""
    s = llsynth.SINGLE_LAYER
    st = Lockstep(ll, 1, s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames,
                  s.chunk_frames, torch.bfloat16)
    ll.ll_set_output_dtype(st.cache, out_dtype)
    if out_dtype == torch.bfloat16:
        st.atol = None  # the bf16 rounding of a value within 1e-2 of the oracle (see compare)
    for c in range(4):  # pre-fill: 12 resident frames
        st.attend(0, *wan_chunk("single", 0, c, s, per_head=True), commit=True, check=False)
    assert st.orc.state(0)[0] == 12
    rows = sample_rows(s.chunk_tokens, 512)
    for p in range(llsynth.SINGLE_LAYER_PASSES):
        q, k, v = wan_chunk("single-pass%d" % p, 0, 4, s, per_head=True)
        st.attend(0, q, k, v, commit=(p == llsynth.SINGLE_LAYER_PASSES - 1), rows=rows,
                  what="single layer pass %d" % p)
        st.check_state()
    st.check_raw(0)  # first eviction: frames 12-14 replaced frames 3-5
    st.close()


def test_stream30_wan(ll):
    s = llsynth.STREAM30
    st = Lockstep(ll, s.layers, s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames,
                  s.chunk_frames, torch.bfloat16)
    checked_layers = (0, 29)
    check_chunks = (0, 3, 4, 5, 19)  # warm-up, last before eviction, first evicting commit, after, last
    rows = sample_rows(s.chunk_tokens, 256)
    for c in range(llsynth.STREAM30_CHUNKS):
        for layer in range(s.layers):
            chunk = wan_chunk("stream30", layer, c, s)
            if layer in checked_layers:
                st.attend(layer, *chunk, commit=True, rows=rows, check=c in check_chunks,
                          what="stream30 L%d c%d" % (layer, c))
            else:
                st.commit_placeholder(layer, *chunk)  # unchecked layer: state only
        st.check_state(layers=checked_layers)
        for layer in (1, 15, 28):
            n, table = ll.ll_cache_state(st.cache, layer)
            assert (n, table) == st.orc.state(layer)
    for layer in checked_layers:
        st.check_raw(layer)
    st.close()


def test_recache30_wan(ll):
    s = llsynth.RECACHE30
    st = Lockstep(ll, s.layers, s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames,
                  s.chunk_frames, torch.bfloat16, keep_frames=False)
    checked_layers = (0, 29)
    rows = sample_rows(s.chunk_tokens, 256)
    R = 12
    prow = sample_rows(R * s.tokens_per_frame, 256, seed=1)
    for c in range(llsynth.RECACHE30_CHUNKS):
        if c in llsynth.RECACHE30_SWITCHES:
            for layer in range(s.layers):
                qw, kw, vw = (llsynth.seeded_normal(("recache30-rc", layer, c, t),
                                                    (R * s.tokens_per_frame, s.heads, s.head_dim), device="cuda")
                              for t in "qkv")
                if layer in checked_layers:
                    st.recache_attend(layer, qw, kw, vw, rows=prow, what="recache30 prefill L%d c%d" % (layer, c))
                else:
                    ll.ll_recache_attend(st.cache, layer, qw, kw, vw, torch.empty_like(qw))
        for layer in range(s.layers):
            chunk = wan_chunk("recache30", layer, c, s)
            if layer in checked_layers:
                st.attend(layer, *chunk, commit=True, rows=rows, check=c in (0, 10, 11, 20, 30, 39),
                          what="recache30 L%d c%d" % (layer, c))
            else:
                st.commit_placeholder(layer, *chunk)
        st.check_state(layers=checked_layers)
    st.close()


SWEEP = [(W, S) for W in llsynth.SWEEP_W for S in llsynth.SWEEP_S]


@pytest.mark.parametrize("W,S", SWEEP, ids=["W%d-S%d" % ws for ws in SWEEP])
def test_sweep_long_horizon(ll, W, S):
    base = llsynth.WAN
    T, C, H, D = base["tokens_per_frame"], base["chunk_frames"], base["heads"], base["head_dim"]
    st = Lockstep(ll, 1, H, D, T, S, W, C, torch.bfloat16, keep_frames=False)
    checks = [c - 1 for c in llsynth.SWEEP_CHECK_CHUNKS]  # 0-based
    # chunks whose frames some check attends to: the sink chunk(s) and the window before each check
    needed = set(checks)
    for c in checks:
        t0 = c * C
        for f in list(range(min(S, t0))) + list(range(max(S, t0 - W), t0)):
            needed.add(f // C)
    rows = sample_rows(C * T, 128)
    shape = llsynth.Shape(1, H, D, T, S, W, C)
    for c in range(llsynth.SWEEP_CHUNKS):
        chunk = wan_chunk(("sweep", W, S), 0, c, shape)
        if c in checks:
            st.attend(0, *chunk, commit=True, rows=rows, what="sweep W%d S%d chunk %d" % (W, S, c + 1))
        elif c in needed:
            st.attend(0, *chunk, commit=True, check=False)
        else:
            st.commit_placeholder(0, *chunk)
        if c in checks or c % 64 == 0:
            st.check_state()
    st.check_state()
    st.close()


def test_long_window_many_keys(ll):
    """A 64-frame window: each chunk attends to 70 frames = 109200 keys (about 850 key tiles per
    work item, 4.7x the longest sweep list); 8 heads x 19 query blocks = 152 items on the SMs,
    so the left-over items are split and merged with very long runs."""
    H, D, T, S, W, C = 8, 128, 1560, 3, 64, 3
    st = Lockstep(ll, 1, H, D, T, S, W, C, torch.bfloat16)
    shape = llsynth.Shape(1, H, D, T, S, W, C)
    n_fill = (S + W) // C + 1
    for c in range(n_fill):  # fill the sink and the window (first evictions included)
        st.attend(0, *wan_chunk("long", 0, c, shape), commit=True, check=False)
    assert st.orc.state(0)[0] == n_fill * C
    rows = sample_rows(C * T, 128, seed=5)
    st.attend(0, *wan_chunk("long-q", 0, n_fill, shape), commit=True, rows=rows, what="long window attend")
    st.check_state()
    st.check_raw(0)
    st.close()


@pytest.mark.parametrize("D", [64, 128])
def test_many_heads_split_tail(ll, D):
    """64 heads of 200-token frames: 64 x 3 = 192 work items of 256 query rows, more than
    the SMs, so an attend launch runs a whole round and then splits the left-over items;
    every row of every pass checked against the oracle, state and slot bytes bit-exact."""
    H, T, S, W, C = 64, 200, 2, 4, 3
    st = Lockstep(ll, 1, H, D, T, S, W, C, torch.bfloat16)
    L = C * T
    for c in range(4):
        q, k, v = (llsynth.seeded_normal(("many-heads", D, c, t), (L, H, D), device="cuda") for t in "qkv")
        st.attend(0, q, k, v, commit=True, what="many heads d%d chunk %d" % (D, c))
        st.check_state()
    st.check_raw(0)
    R = len(st.orc.recache_frames(0))
    qw, kw, vw = (llsynth.seeded_normal(("many-heads-rc", D, t), (R * T, H, D), device="cuda") for t in "qkv")
    st.recache_attend(0, qw, kw, vw, what="many heads d%d prefill" % D)
    st.check_state()
    st.check_raw(0)
    st.close()
