"""Pins of the oracle's two optional readings: the frame-causal chunk mask and the
keep-sink recache scope ("LongLive", §3.3: the model is frame-level
autoregressive, and the recache rebuilds the cache only from the most recent W
frames).

As in test_oracle_pins.py, every check rests on something other than the
oracle's own formulas: a hand-written golden table (tests/golden/), scalar loops
over key lists the test assembles itself, torch's scaled_dot_product_attention in
float64, invariants (one-frame chunks, last-frame rows, recache-then-attend), and
planted mistakes that the pins must catch.
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import ll_oracle as O
from tests.conftest import read_golden

H, D, T = 1, 2, 2


def frame_code_chunk(f0, C, T_, H_, D_):
    """[C*T, H, D] with every token of frame f0 + i set to the code f0 + i."""
    x = np.zeros((C * T_, H_, D_))
    for i in range(C):
        x[i * T_:(i + 1) * T_] = f0 + i
    return x


def committed_cache(S, W, C, n, **opts):
    """A cache whose committed frames carry V = frame code, K = 0."""
    c = O.OracleCache(1, H, D, T, S, W, C, **opts)
    while c.layers[0].n < n:
        f0 = c.layers[0].n
        z = np.zeros((C * T, H, D))
        c.attend(0, z, z, frame_code_chunk(f0, C, T, H, D), commit=True)
    return c


def probe(mode, S, W, C, t0, qframe):
    """Output code of query frame qframe under `mode` (see the golden file)."""
    if mode == "attend-frame":
        c = committed_cache(S, W, C, t0, chunk_mask="frame")
        z = np.zeros((C * T, H, D))
        out = c.attend(0, z, z, frame_code_chunk(t0, C, T, H, D), commit=False)
        row = (qframe - t0) * T
        return out[row:row + T]
    scope, mask = {"prefill-window-chunk": ("window", "chunk"), "prefill-window-frame": ("window", "frame"),
                   "prefill-resident-frame": ("resident", "frame")}[mode]
    c = committed_cache(S, W, C, t0, chunk_mask=mask, recache_scope=scope)
    frames = c.recache_frames(0)
    L = len(frames) * T
    v = np.zeros((L, H, D))
    for i, f in enumerate(frames):
        v[i * T:(i + 1) * T] = f
    z = np.zeros((L, H, D))
    out = c.recache_attend(0, z, z, v)
    row = frames.index(qframe) * T
    return out[row:row + T]


def golden_mismatches():
    bad = []
    for left, right in read_golden("variant_visible_means.txt"):
        mode = left[0]
        S, W, C, t0, qframe = map(int, left[1:])
        want = float(Fraction(right[0]))
        got = probe(mode, S, W, C, t0, qframe)
        if not np.allclose(got, want, rtol=0, atol=1e-12):
            bad.append((mode, S, W, C, t0, qframe, float(got.ravel()[0]), want))
    return bad


def test_variant_visibility_golden():
    assert golden_mismatches() == []


# ---------------------------------------------------------------------------
# Frame-causal chunk mask
# ---------------------------------------------------------------------------


def frame_mask_brute_force_mismatch(seed=0):
    """Scalar float64 loops over the key list each query row may see, assembled here
    from the frames this test committed (sink, last-W window, chunk frames up to the
    query's own frame)."""
    rng = np.random.default_rng(seed)
    S, W, C, T_, H_, D_ = 2, 3, 3, 2, 2, 4
    c = O.OracleCache(1, H_, D_, T_, S, W, C, chunk_mask="frame")
    frames = {}
    worst = 0.0
    for chunk in range(4):
        t0 = chunk * C
        q, k, v = (rng.standard_normal((C * T_, H_, D_)) for _ in range(3))
        got = c.attend(0, q, k, v, commit=True)
        for i in range(C):
            frames[t0 + i] = (k[i * T_:(i + 1) * T_], v[i * T_:(i + 1) * T_])
        cached = [f for f in range(t0) if f < S or f >= max(S, t0 - W)]
        for row in range(C * T_):
            own = t0 + row // T_
            keys = [frames[f] for f in cached + list(range(t0, own + 1))]
            for h in range(H_):
                kk = [kf[tok, h] for kf, _ in keys for tok in range(T_)]
                vv = [vf[tok, h] for _, vf in keys for tok in range(T_)]
                s = [sum(q[row, h, e] * kj[e] for e in range(D_)) / math.sqrt(D_) for kj in kk]
                mx = max(s)
                wts = [math.exp(x - mx) for x in s]
                tot = sum(wts)
                for e in range(D_):
                    want = sum(wj * vj[e] for wj, vj in zip(wts, vv)) / tot
                    worst = max(worst, abs(got[row, h, e] - want))
    return worst


def test_frame_mask_brute_force():
    assert frame_mask_brute_force_mismatch() < 1e-12


def test_frame_mask_equals_chunk_mask_for_one_frame_chunks():
    rng = np.random.default_rng(1)
    S, W, C = 1, 3, 1
    a = O.OracleCache(1, H, D, T, S, W, C, chunk_mask="chunk")
    b = O.OracleCache(1, H, D, T, S, W, C, chunk_mask="frame")
    for _ in range(6):
        q, k, v = (rng.standard_normal((C * T, H, D)) for _ in range(3))
        assert np.array_equal(a.attend(0, q, k, v, commit=True), b.attend(0, q, k, v, commit=True))
    kw, vw, qw = (rng.standard_normal((len(a.resident(0)) * T, H, D)) for _ in range(3))
    assert np.array_equal(a.recache_attend(0, qw, kw, vw), b.recache_attend(0, qw, kw, vw))


def test_frame_mask_last_frame_rows_equal_chunk_mask():
    """The chunk's last frame sees the whole chunk under either mask."""
    rng = np.random.default_rng(2)
    S, W, C, T_ = 2, 4, 3, 3
    a = O.OracleCache(1, 2, 4, T_, S, W, C)
    b = O.OracleCache(1, 2, 4, T_, S, W, C, chunk_mask="frame")
    for _ in range(4):
        q, k, v = (rng.standard_normal((C * T_, 2, 4)) for _ in range(3))
        oa = a.attend(0, q, k, v, commit=True)
        ob = b.attend(0, q, k, v, commit=True)
        last = slice((C - 1) * T_, C * T_)
        np.testing.assert_allclose(ob[last], oa[last], rtol=0, atol=1e-13)
        assert not np.allclose(ob[:T_], oa[:T_])  # the first frame sees less


# ---------------------------------------------------------------------------
# Keep-sink recache scope
# ---------------------------------------------------------------------------


def filled(rng, S, W, C, n, **opts):
    c = O.OracleCache(1, H, D, T, S, W, C, **opts)
    while c.layers[0].n < n:
        q, k, v = (rng.standard_normal((C * T, H, D)) for _ in range(3))
        c.attend(0, q, k, v, commit=True)
    return c


def keep_sink_state_ok():
    rng = np.random.default_rng(3)
    S, W, C, n = 3, 6, 3, 15
    c = filled(rng, S, W, C, n, recache_scope="window")
    before = {f: (kv[0].copy(), kv[1].copy()) for f, kv in c.layers[0].frames.items()}
    table = c.state(0)
    window = [f for f in range(n) if f >= max(S, n - W)]
    kw, vw = (rng.standard_normal((len(window) * T, H, D)) for _ in range(2))
    c.recache(0, kw, vw)
    if c.state(0) != table:
        return False
    for f in range(S):  # sink untouched
        if not (np.array_equal(c.frame_kv(0, f)[0], before[f][0]) and np.array_equal(c.frame_kv(0, f)[1], before[f][1])):
            return False
    for i, f in enumerate(window):  # window replaced, in list order
        if not (np.array_equal(c.frame_kv(0, f)[0], kw[i * T:(i + 1) * T]) and
                np.array_equal(c.frame_kv(0, f)[1], vw[i * T:(i + 1) * T])):
            return False
    return True


def test_keep_sink_recache_state():
    assert keep_sink_state_ok()


def keep_sink_prefill_sdpa_err(block_frames_mask="chunk"):
    """The keep-sink prefill against torch SDPA (float64) with an explicit mask built here."""
    rng = np.random.default_rng(4)
    S, W, C, n, H_, D_ = 2, 5, 3, 12, 2, 8
    c = O.OracleCache(1, H_, D_, T, S, W, C, recache_scope="window", chunk_mask=block_frames_mask)
    while c.layers[0].n < n:
        q, k, v = (rng.standard_normal((C * T, H_, D_)) for _ in range(3))
        c.attend(0, q, k, v, commit=True)
    sink = list(range(S))
    window = list(range(max(S, n - W), n))
    Ks = np.concatenate([c.frame_kv(0, f)[0] for f in sink])
    Vs = np.concatenate([c.frame_kv(0, f)[1] for f in sink])
    Lw = len(window) * T
    qw, kw, vw = (rng.standard_normal((Lw, H_, D_)) for _ in range(3))
    got = c.recache_attend(0, qw, kw, vw)
    bf = C if block_frames_mask == "chunk" else 1
    mask = np.zeros((Lw, len(sink) * T + Lw), dtype=bool)
    for qi in range(Lw):
        mask[qi, :len(sink) * T] = True
        for kj in range(Lw):
            mask[qi, len(sink) * T + kj] = (kj // T) // bf <= (qi // T) // bf
    K = np.concatenate([Ks, kw])
    V = np.concatenate([Vs, vw])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qw).permute(1, 0, 2), torch.from_numpy(K).permute(1, 0, 2),
        torch.from_numpy(V).permute(1, 0, 2), attn_mask=torch.from_numpy(mask)).permute(1, 0, 2).numpy()
    return float(np.abs(got - ref).max())


@pytest.mark.parametrize("mask", ["chunk", "frame"])
def test_keep_sink_prefill_matches_sdpa(mask):
    assert keep_sink_prefill_sdpa_err(mask) < 1e-12


def keep_sink_recache_then_attend_err():
    """recache(window) then attend == attend on a cache committed with (old sink, new window)."""
    rng = np.random.default_rng(5)
    S, W, C = 3, 6, 3
    n = S + W  # nothing evicted yet: every non-sink frame is in the window
    chunks = [tuple(rng.standard_normal((C * T, H, D)) for _ in range(3)) for _ in range(n // C)]
    a = O.OracleCache(1, H, D, T, S, W, C, recache_scope="window")
    for q, k, v in chunks:
        a.attend(0, q, k, v, commit=True)
    kw, vw = (rng.standard_normal(((n - S) * T, H, D)) for _ in range(2))
    a.recache(0, kw, vw)
    b = O.OracleCache(1, H, D, T, S, W, C)
    for ci, (q, k, v) in enumerate(chunks):
        k2, v2 = k.copy(), v.copy()
        for i in range(C):
            f = ci * C + i
            if f >= S:
                k2[i * T:(i + 1) * T] = kw[(f - S) * T:(f - S + 1) * T]
                v2[i * T:(i + 1) * T] = vw[(f - S) * T:(f - S + 1) * T]
        b.attend(0, q, k2, v2, commit=True)
    q, k, v = (rng.standard_normal((C * T, H, D)) for _ in range(3))
    return float(np.abs(a.attend(0, q, k, v, commit=False) - b.attend(0, q, k, v, commit=False)).max())


def test_keep_sink_recache_then_attend_equals_from_scratch():
    assert keep_sink_recache_then_attend_err() == 0.0


def test_keep_sink_recache_of_a_layer_without_window_is_rejected():
    rng = np.random.default_rng(6)
    c = filled(rng, 3, 6, 3, 3, recache_scope="window")  # only the sink is resident
    assert c.recache_frames(0) == []
    with pytest.raises(ValueError):
        c.recache(0, np.zeros((0, H, D)), np.zeros((0, H, D)))


# ---------------------------------------------------------------------------
# Planted mistakes: each must make at least one of the pins above fail
# ---------------------------------------------------------------------------


def all_variant_pins_pass():
    try:
        return (golden_mismatches() == [] and frame_mask_brute_force_mismatch() < 1e-12 and keep_sink_state_ok()
                and keep_sink_prefill_sdpa_err("chunk") < 1e-12 and keep_sink_prefill_sdpa_err("frame") < 1e-12
                and keep_sink_recache_then_attend_err() == 0.0)
    except (AssertionError, ValueError, IndexError, KeyError):
        return False


def _strict_block(n_prefix, block_tokens, Lkv):
    # off by one: a query does not see its own block
    kj = np.arange(Lkv)
    after = kj >= n_prefix
    kb = np.where(after, (kj - n_prefix) // block_tokens, -1)
    return lambda qi: ~after | (kb < (qi // block_tokens))


def _prefix_hidden(n_prefix, block_tokens, Lkv):
    # the cached prefix is masked like the chunk instead of fully visible
    kb = np.arange(Lkv) // block_tokens
    return lambda qi: kb <= (qi // block_tokens)


def _recache_frames_with_sink(self, layer):
    # keep-sink scope that rewrites the sink as well
    return O.resident_frames(self.S, self.W, self.layers[layer].n)


def _chunk_blocks_for_frame_mask(self):
    # frame mask that still uses C-frame blocks in the prefill
    return self.C


PLANTED = [
    ("block mask excludes its own block", O, "prefix_then_block_causal_visible", _strict_block),
    ("cached prefix masked", O, "prefix_then_block_causal_visible", _prefix_hidden),
    ("keep-sink recache rewrites the sink", O.OracleCache, "recache_frames", _recache_frames_with_sink),
    ("frame-mask prefill in chunk blocks", O.OracleCache, "_block_frames", _chunk_blocks_for_frame_mask),
]


def test_variant_pins_pass_unplanted():
    assert all_variant_pins_pass()


@pytest.mark.parametrize("name,owner,target,fake", PLANTED, ids=[p[0] for p in PLANTED])
def test_planted_variant_mistakes_are_caught(monkeypatch, name, owner, target, fake):
    monkeypatch.setattr(owner, target, fake)
    assert not all_variant_pins_pass(), "planted mistake not caught: " + name
