"""Pins of the float64 oracle against facts that do not come from the oracle itself.

Each check uses something independent of the oracle's own formulas: hand-written
golden tables (tests/golden/), brute-force scalar loops, a library routine
(torch's scaled_dot_product_attention in float64 on the CPU), closed forms and
invariants.  ``test_planted_mistakes_are_caught`` plants plausible mistakes in
the oracle (on the CPU) and checks that these pins catch each of them.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import ll_oracle as O
from tests.conftest import read_golden


def rnd(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


# ---------------------------------------------------------------------------
# Cache bookkeeping: hand-written golden tables
# ---------------------------------------------------------------------------


def check_slot_maps():
    bad = []
    for left, right in read_golden("slot_maps.txt"):
        S, W, C, n = map(int, left)
        want = [int(x) for x in right]
        c = O.OracleCache(1, 1, 1, 1, S, W, C)
        T = 1
        while c.layers[0].n < n:
            z = np.zeros((C * T, 1, 1))
            c.attend(0, z, z, z, commit=True)
        got = c.state(0)[1]
        if got != want or c.state(0)[0] != n:
            bad.append((S, W, C, n, got, want))
    return bad


def test_slot_maps_golden():
    assert check_slot_maps() == []


def test_slot_map_is_a_bijection_of_resident_frames():
    for S in range(0, 5):
        for W in range(0, 7):
            for C in range(1, 5):
                for n in range(0, 40, C):
                    table = O.frame_of_slot(S, W, n)
                    occupied = sorted(f for f in table if f >= 0)
                    assert occupied == O.resident_frames(S, W, n)
                    # sink frames never move; ring frames keep their slot until evicted
                    for f in occupied:
                        if f < S:
                            assert table[f] == f


def test_visible_counts_closed_form():
    # sink + window + chunk, in frames, for the Wan-shaped cache (S=3, W=9, C=3):
    # warm-up chunks see 3, 6, 9, 12 frames, then a steady 15 frames = 23400 tokens.
    S, W, C, T = 3, 9, 3, 1560
    want = {0: 3, 3: 6, 6: 9, 9: 12, 12: 15, 15: 15, 300: 15}
    for t0, frames in want.items():
        assert len(O.visible_frames(S, W, C, t0)) == frames
        assert O.lkv_tokens(S, W, C, T, t0) == frames * T
    assert O.lkv_tokens(S, W, C, T, 12) == 23400


def test_tokens_per_frame_closed_form():
    # 832x480 video ("LongLive", §4 Implementation) -> 8x spatial VAE and 2x2
    # patches (Wan2.1) -> a 30x52 grid = 1560 tokens per latent frame.  §1 says a
    # 180 s Wan-2.1 video is over a million tokens: 180 s x 16 FPS = 2880 frames,
    # 4x temporal VAE compression (+1 leading frame) -> 721 latent frames.
    T = (480 // 16) * (832 // 16)
    assert T == 1560
    latent = 1 + (180 * 16 - 1) // 4 + 1
    assert latent * T > 1_000_000


# ---------------------------------------------------------------------------
# Attention arithmetic
# ---------------------------------------------------------------------------


def brute_force_row(q_row, K, V):
    """softmax(q k / sqrt(d)) V for one query row, scalar loops in pure Python."""
    d = len(q_row)
    scores = []
    for j in range(len(K)):
        s = 0.0
        for t in range(d):
            s += q_row[t] * K[j][t]
        scores.append(s / math.sqrt(d))
    m = max(scores)
    w = [math.exp(s - m) for s in scores]
    z = sum(w)
    return [sum(w[j] * V[j][t] for j in range(len(K))) / z for t in range(d)]


def test_masked_attention_brute_force():
    rng = np.random.default_rng(1)
    q, k, v = rnd(rng, 5, 2, 8), rnd(rng, 7, 2, 8), rnd(rng, 7, 2, 8)
    out = O.masked_attention(q, k, v)
    for i in range(5):
        for h in range(2):
            want = brute_force_row(list(q[i, h]), [list(r) for r in k[:, h]], [list(r) for r in v[:, h]])
            np.testing.assert_allclose(out[i, h], want, rtol=1e-12, atol=1e-12)


def sdpa64(q, k, v, mask=None):
    """torch's scaled_dot_product_attention on the CPU in float64; [L, H, d] layout."""
    tq = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))
    tk = torch.from_numpy(np.ascontiguousarray(k.transpose(1, 0, 2)))
    tv = torch.from_numpy(np.ascontiguousarray(v.transpose(1, 0, 2)))
    m = None if mask is None else torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m)
    return o.numpy().transpose(1, 0, 2)


def run_chunks(cache, chunks, layer=0):
    """Attend + commit each (q, k, v) chunk in turn; returns the outputs."""
    return [cache.attend(layer, q, k, v, commit=True) for (q, k, v) in chunks]


def make_chunks(rng, n, L, H, d):
    return [tuple(rnd(rng, L, H, d, scale=0.5) for _ in range(3)) for _ in range(n)]


def check_no_sink_no_window():
    """S = W = 0: every chunk is plain self-attention over its own tokens."""
    rng = np.random.default_rng(2)
    T, C, H, d = 4, 3, 2, 8
    cache = O.OracleCache(1, H, d, T, 0, 0, C)
    chunks = make_chunks(rng, 4, C * T, H, d)
    outs = run_chunks(cache, chunks)
    return max(float(np.abs(o - sdpa64(q, k, v)).max()) for o, (q, k, v) in zip(outs, chunks))


def test_no_sink_no_window_is_chunk_self_attention():
    assert check_no_sink_no_window() < 1e-12


def check_full_history():
    """W covering the whole history: block-causal full attention over all frames."""
    rng = np.random.default_rng(3)
    T, C, H, d, S = 3, 2, 2, 8, 2
    cache = O.OracleCache(1, H, d, T, S, 100, C)
    chunks = make_chunks(rng, 5, C * T, H, d)
    outs = run_chunks(cache, chunks)
    err = 0.0
    for c, (q, _, _) in enumerate(chunks):
        K = np.concatenate([ch[1] for ch in chunks[:c + 1]])
        V = np.concatenate([ch[2] for ch in chunks[:c + 1]])
        err = max(err, float(np.abs(outs[c] - sdpa64(q, K, V)).max()))
    return err


def test_full_window_is_block_causal_full_attention():
    assert check_full_history() < 1e-12


def check_window_by_library():
    """S=3, W=6, C=3: each chunk = textbook attention over its hand-listed frames."""
    rng = np.random.default_rng(4)
    T, C, H, d, S, W = 2, 3, 2, 8, 3, 6
    cache = O.OracleCache(1, H, d, T, S, W, C)
    chunks = make_chunks(rng, 8, C * T, H, d)
    outs = run_chunks(cache, chunks)
    # frames visible to chunk c (t0 = 3c), written out by hand from §3.3
    visible = {0: [0, 1, 2], 1: [0, 1, 2, 3, 4, 5], 2: list(range(9)), 3: list(range(12)),
               4: [0, 1, 2] + list(range(6, 15)), 5: [0, 1, 2] + list(range(9, 18)),
               6: [0, 1, 2] + list(range(12, 21)), 7: [0, 1, 2] + list(range(15, 24))}
    err = 0.0
    for c, (q, _, _) in enumerate(chunks):
        def frame_rows(t, f):
            ch, i = divmod(f, C)
            return chunks[ch][t][i * T:(i + 1) * T]
        K = np.concatenate([frame_rows(1, f) for f in visible[c]])
        V = np.concatenate([frame_rows(2, f) for f in visible[c]])
        err = max(err, float(np.abs(outs[c] - sdpa64(q, K, V)).max()))
    return err


def test_window_and_sink_against_library_attention():
    assert check_window_by_library() < 1e-12


def check_visible_means():
    bad = []
    for left, right in read_golden("visible_means.txt"):
        S, W, C, t0 = map(int, left)
        want = float(right[0])
        T, H, d = 2, 2, 4
        cache = O.OracleCache(1, H, d, T, S, W, C)
        for c in range(t0 // C + 1):
            codes = np.repeat(np.arange(c * C, (c + 1) * C, dtype=np.float64), T)
            v = np.broadcast_to(codes[:, None, None], (C * T, H, d)).copy()
            z = np.zeros((C * T, H, d))
            out = cache.attend(0, z, np.ones((C * T, H, d)), v, commit=(c < t0 // C))
        if abs(float(out.max()) - want) > 1e-12 or abs(float(out.min()) - want) > 1e-12:
            bad.append((S, W, C, t0, float(out.mean()), want))
    return bad


def test_visibility_probe_golden():
    assert check_visible_means() == []


def test_softmax_invariants():
    rng = np.random.default_rng(5)
    q, k = rnd(rng, 6, 3, 8), rnd(rng, 9, 3, 8)
    # V = c everywhere -> O = c; V = 1 -> the weights of each row sum to 1
    np.testing.assert_allclose(O.masked_attention(q, k, np.full((9, 3, 8), 2.5)), 2.5, rtol=1e-13)
    # permuting the key/value list leaves every output unchanged
    v = rnd(rng, 9, 3, 8)
    perm = rng.permutation(9)
    np.testing.assert_allclose(O.masked_attention(q, k, v), O.masked_attention(q, k[perm], v[perm]),
                               rtol=1e-12, atol=1e-13)
    # a sampled row subset equals the same rows of the full result
    np.testing.assert_allclose(O.masked_attention(q, k, v, rows=[4, 1]), O.masked_attention(q, k, v)[[4, 1]],
                               rtol=0, atol=0)


def test_only_commit_pass_mutates_state():
    rng = np.random.default_rng(6)
    T, C, H, d = 2, 3, 1, 4
    cache = O.OracleCache(1, H, d, T, 3, 6, C)
    ch = make_chunks(rng, 3, C * T, H, d)
    a = cache.attend(0, *ch[0], commit=False)
    assert cache.state(0)[0] == 0
    b = cache.attend(0, *ch[0], commit=True)
    np.testing.assert_array_equal(a, b)
    assert cache.state(0)[0] == 3
    cache.reset()
    assert cache.state(0) == (0, [-1] * 9)


# ---------------------------------------------------------------------------
# Recache
# ---------------------------------------------------------------------------


def check_recache_equals_scratch():
    """Recache then attend == a fresh cache whose resident frames hold the recache K/V."""
    rng = np.random.default_rng(7)
    T, C, H, d, S, W = 2, 3, 2, 8, 3, 6
    a = O.OracleCache(1, H, d, T, S, W, C)
    run_chunks(a, make_chunks(rng, 5, C * T, H, d))          # n = 15: frames 0-2, 9-14 resident
    k_win, v_win = rnd(rng, 9 * T, H, d), rnd(rng, 9 * T, H, d)
    a.recache(0, k_win, v_win)
    q_next, k_next, v_next = (rnd(rng, C * T, H, d) for _ in range(3))
    out_a = a.attend(0, q_next, k_next, v_next, commit=False)
    # from scratch: chunk 0 carries the sink part of the recache K/V, chunks 3 and 4
    # the window part; chunks 1 and 2 are evicted by n = 15 and may hold anything.
    b = O.OracleCache(1, H, d, T, S, W, C)
    filler = make_chunks(rng, 2, C * T, H, d)
    z = np.zeros((C * T, H, d))
    b.attend(0, z, k_win[0:3 * T], v_win[0:3 * T], commit=True)
    for ch in filler:
        b.attend(0, *ch, commit=True)
    b.attend(0, z, k_win[3 * T:6 * T], v_win[3 * T:6 * T], commit=True)
    b.attend(0, z, k_win[6 * T:9 * T], v_win[6 * T:9 * T], commit=True)
    out_b = b.attend(0, q_next, k_next, v_next, commit=False)
    assert a.state(0) == b.state(0)
    return float(np.abs(out_a - out_b).max())


def test_recache_then_attend_equals_scratch():
    assert check_recache_equals_scratch() < 1e-12


def test_recache_keeps_frame_indices_and_empty_recache_fails():
    rng = np.random.default_rng(8)
    T, C, H, d = 2, 3, 1, 4
    cache = O.OracleCache(1, H, d, T, 3, 6, C)
    with pytest.raises(ValueError):
        cache.recache(0, np.zeros((0, H, d)), np.zeros((0, H, d)))
    run_chunks(cache, make_chunks(rng, 4, C * T, H, d))
    before = cache.state(0)
    cache.recache(0, rnd(rng, 9 * T, H, d), rnd(rng, 9 * T, H, d))
    assert cache.state(0) == before


def check_prefill_block_causal():
    """Prefill output of list block g == textbook attention over list blocks 0..g."""
    rng = np.random.default_rng(9)
    T, C, H, d, S, W = 2, 3, 2, 8, 3, 9
    cache = O.OracleCache(1, H, d, T, S, W, C)
    run_chunks(cache, make_chunks(rng, 6, C * T, H, d))       # 12 resident frames: 4 blocks
    R = 12
    qw, kw, vw = (rnd(rng, R * T, H, d) for _ in range(3))
    out = cache.recache_attend(0, qw, kw, vw)
    bt = C * T
    err = 0.0
    for g in range(R // C):
        rows = slice(g * bt, (g + 1) * bt)
        want = sdpa64(qw[rows], kw[:(g + 1) * bt], vw[:(g + 1) * bt])
        err = max(err, float(np.abs(out[rows] - want).max()))
    return err


def test_prefill_is_block_causal_over_the_list():
    assert check_prefill_block_causal() < 1e-12


def test_prefill_ragged_last_block():
    # R = 7 frames with C = 3: blocks of 3, 3 and 1 frame
    rng = np.random.default_rng(10)
    T, C, H, d = 2, 3, 1, 4
    cache = O.OracleCache(1, H, d, T, 3, 4, C)
    run_chunks(cache, make_chunks(rng, 3, C * T, H, d))       # n = 9: frames 0-2 and 5-8
    assert len(cache.resident(0)) == 7
    qw, kw, vw = (rnd(rng, 7 * T, H, d) for _ in range(3))
    out = cache.recache_attend(0, qw, kw, vw)
    np.testing.assert_allclose(out[12:14], sdpa64(qw[12:14], kw, vw), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out[6:12], sdpa64(qw[6:12], kw[:12], vw[:12]), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------


def all_pins_pass():
    try:
        ok = (check_slot_maps() == [] and check_visible_means() == []
              and check_no_sink_no_window() < 1e-12 and check_full_history() < 1e-12
              and check_window_by_library() < 1e-12 and check_recache_equals_scratch() < 1e-12
              and check_prefill_block_causal() < 1e-12)
    except (AssertionError, ValueError, KeyError, IndexError):
        ok = False
    return ok


def _window_off_by_one(S, W, n):
    lo = max(S, n - W + 1)
    return list(range(lo, n)) if n > lo else []


def _window_overlaps_sink(S, W, n):
    lo = max(0, n - W)
    return list(range(lo, n)) if n > lo else []


def _slot_without_offset(S, W, f):
    return f if f < S else (f % (S + W))


def _sink_dropped(S, n):
    return []


def _scale_missing(q, k, v, visible=None, rows=None, block_rows=512):
    return _orig_masked(q * math.sqrt(q.shape[-1]), k, v, visible, rows, block_rows)


def _causal_mask_strict(T, C, Lkv):
    bt = C * T
    kb = np.arange(Lkv) // bt
    return lambda qi: kb < (qi // bt) + (1 if qi % bt else 0)


_orig_masked = O.masked_attention


@pytest.mark.parametrize("name,target,fake", [
    ("window off by one", "window_frames", _window_off_by_one),
    ("window overlaps sink", "window_frames", _window_overlaps_sink),
    ("ring slot without sink offset", "slot_of_frame", _slot_without_offset),
    ("sink dropped", "sink_frames", _sink_dropped),
    ("missing 1/sqrt(d)", "masked_attention", _scale_missing),
    ("wrong prefill mask", "block_causal_visible", _causal_mask_strict),
])
def test_planted_mistakes_are_caught(monkeypatch, name, target, fake):
    assert all_pins_pass()
    monkeypatch.setattr(O, target, fake)
    assert not all_pins_pass(), "planted mistake not caught: " + name


def test_oracle_package_exports():
    assert oracle.OracleCache is O.OracleCache
