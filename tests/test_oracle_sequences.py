"""Pin of the oracle on random call sequences against a full-history brute force.

The model here keeps every frame ever committed (it evicts nothing) and, at
each call, decides per key whether the query may see it, straight from the
definition of the method (LongLive §3.3 "Frame sink" + "Short window
attention", §3.1 "KV recache"; §4.4 Table 4 for the reset):

* a query of the chunk starting at frame t0 sees the sink frames f < min(S, t0),
  the window frames max(S, t0 - W) <= f < t0 and the chunk's own frames (all of
  them, or with the frame mask those up to its own frame);
* a recache rewrites the K/V of the frames that such a query would see from the
  cache (with the keep-sink scope only the window frames), and its prefill
  queries see the rewritten frames block-causally by their position in that
  list (and, with the keep-sink scope, every sink frame's cached K/V).

A frame that has left the window never returns to it (t0 only grows), so this
model needs no eviction at all, whereas the oracle deletes frames as they fall
out of the window.  Attention is computed with scalar loops in pure Python.
"""

import math

import numpy as np
import pytest

from oracle import ll_oracle as O

CASES = 300


def brute_attention(q_rows, keys, visible):
    """q_rows: list of (query frame, [H][d] vector); keys: list of (key frame, K [H][d], V [H][d]);
    visible(query frame, key frame) -> bool.  Returns [rows][H][d] as nested lists."""
    out = []
    for qf, q in q_rows:
        per_head = []
        for h in range(len(q)):
            d = len(q[h])
            scores, vals = [], []
            for kf, K, V in keys:
                if visible(qf, kf):
                    scores.append(sum(q[h][i] * K[h][i] for i in range(d)) / math.sqrt(d))
                    vals.append(V[h])
            m = max(scores)
            w = [math.exp(s - m) for s in scores]
            tot = sum(w)
            per_head.append([sum(w[j] * vals[j][i] for j in range(len(w))) / tot for i in range(d)])
        out.append(per_head)
    return out


class History:
    def __init__(self, S, W, C, T):
        self.S, self.W, self.C, self.T = S, W, C, T
        self.frames = {}  # frame -> (K [T][H][d], V [T][H][d]) as nested lists
        self.n = 0
        self.mask, self.scope = "chunk", "resident"

    def _cached(self, t0):
        return [f for f in sorted(self.frames)
                if f < min(self.S, t0) or max(self.S, t0 - self.W) <= f < t0]

    def attend(self, q, k, v, commit):
        T, t0 = self.T, self.n
        keys = [(f, self.frames[f][0][r], self.frames[f][1][r]) for f in self._cached(t0) for r in range(T)]
        keys += [(t0 + r // T, k[r], v[r]) for r in range(len(k))]
        q_rows = [(t0 + r // T, q[r]) for r in range(len(q))]
        frame_mask = self.mask == "frame"
        out = brute_attention(q_rows, keys, lambda qf, kf: kf < t0 or not frame_mask or kf <= qf)
        if commit:
            for i in range(self.C):
                self.frames[t0 + i] = (k[i * T:(i + 1) * T], v[i * T:(i + 1) * T])
            self.n = t0 + self.C
        return out

    def recache_list(self):
        listed = self._cached(self.n)
        if self.scope == "window":
            listed = [f for f in listed if f >= self.S]
        return listed

    def recache(self, k, v, q=None):
        T = self.T
        listed = self.recache_list()
        block = 1 if self.mask == "frame" else self.C
        out = None
        if q is not None:
            # keys carry their list position (fresh frames) or -1 (cached sink frames)
            keys = [(p, k[p * T + r], v[p * T + r]) for p in range(len(listed)) for r in range(T)]
            if self.scope == "window":
                sink = [f for f in self._cached(self.n) if f < self.S]
                keys = [(-1, self.frames[f][0][r], self.frames[f][1][r]) for f in sink for r in range(T)] + keys
            q_rows = [(r // T, q[r]) for r in range(len(q))]
            out = brute_attention(q_rows, keys, lambda qp, kp: kp < 0 or kp // block <= qp // block)
        for p, f in enumerate(listed):
            self.frames[f] = (k[p * T:(p + 1) * T], v[p * T:(p + 1) * T])
        return out


def sequence_passes(seed):
    """Run one random call sequence on the oracle and the full-history model; True when
    every output matches to 1e-10 and the committed counts and recached lists agree."""
    rng = np.random.default_rng(5000 + seed)
    S, W, C, T = int(rng.integers(0, 4)), int(rng.integers(0, 6)), int(rng.integers(1, 4)), int(rng.integers(1, 4))
    H, d = int(rng.integers(1, 3)), int(rng.choice([2, 4]))
    orc = O.OracleCache(1, H, d, T, S, W, C)
    ref = History(S, W, C, T)
    ops = ["commit"] * 4 + ["pass"] * 2 + ["prefill", "recache", "reset", "options"]

    def draw(rows):
        return rng.standard_normal((rows, H, d))

    try:
        for _ in range(int(rng.integers(15, 31))):
            op = str(rng.choice(ops))
            if op in ("commit", "pass"):
                q, k, v = draw(C * T), draw(C * T), draw(C * T)
                got = orc.attend(0, q, k, v, commit=(op == "commit"))
                want = ref.attend(q.tolist(), k.tolist(), v.tolist(), op == "commit")
                if np.abs(got - np.array(want)).max() > 1e-10:
                    return False
            elif op in ("prefill", "recache"):
                listed = ref.recache_list()
                if orc.recache_frames(0) != listed:
                    return False
                if not listed:
                    try:
                        orc.recache(0, np.zeros((0, H, d)), np.zeros((0, H, d)))
                    except ValueError:
                        continue
                    return False
                R = len(listed)
                q, k, v = draw(R * T), draw(R * T), draw(R * T)
                if op == "prefill":
                    got = orc.recache_attend(0, q, k, v)
                    want = ref.recache(k.tolist(), v.tolist(), q.tolist())
                    if np.abs(got - np.array(want)).max() > 1e-10:
                        return False
                else:
                    orc.recache(0, k, v)
                    ref.recache(k.tolist(), v.tolist())
            elif op == "reset":
                orc.reset()
                ref.frames, ref.n = {}, 0
            else:
                ref.mask = str(rng.choice(["chunk", "frame"]))
                ref.scope = str(rng.choice(["resident", "window"]))
                orc.set_chunk_mask(ref.mask)
                orc.set_recache_scope(ref.scope)
            if orc.state(0)[0] != ref.n:
                return False
    except (AssertionError, ValueError, KeyError, IndexError):
        return False
    return True


@pytest.mark.parametrize("block", range(CASES // 50))
def test_oracle_matches_full_history_brute_force(block):
    failed = [seed for seed in range(50 * block, 50 * block + 50) if not sequence_passes(seed)]
    assert failed == []


def _window_one_late(S, W, n):
    lo = max(S, n - W - 1)
    return list(range(lo, n)) if n > lo else []


def _reset_keeps_count(self):
    for lay in self.layers:
        lay.frames.clear()


def _recache_list_reversed(self, layer):
    return list(reversed(_orig_recache_frames(self, layer)))


def _frame_mask_ignored(n_prefix, block_tokens, Lkv):
    return lambda qi: np.ones(Lkv, dtype=bool)


_orig_recache_frames = O.OracleCache.recache_frames


@pytest.mark.parametrize("name,owner,attr,fake", [
    ("eviction one frame late", O, "window_frames", _window_one_late),
    ("reset keeps the committed count", O.OracleCache, "reset", _reset_keeps_count),
    ("recache list reversed", O.OracleCache, "recache_frames", _recache_list_reversed),
    ("frame mask ignored", O, "prefix_then_block_causal_visible", _frame_mask_ignored),
])
def test_planted_sequence_mistakes_are_caught(monkeypatch, name, owner, attr, fake):
    seeds = range(60)
    assert all(sequence_passes(s) for s in seeds)
    monkeypatch.setattr(owner, attr, fake)
    assert not all(sequence_passes(s) for s in seeds), "planted mistake not caught: " + name
