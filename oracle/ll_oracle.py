"""Float64 CPU oracle for short-window + frame-sink attention over a rolling KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library and imports nothing from it.

Source: "LongLive: Real-time Interactive Long Video Generation" (Chinese
translation of the paper body on gitcode.csdn.net, and the course.zhidx.com
digest of it).  Every function below names the passage it restates.

What the method computes (the plain definition this module writes out):

* §3.3 "Short window attention": each generation step attends only to a fixed
  temporal window of the most recent W latent frames; the per-layer KV cache
  holds those frames, not the whole video.
* §3.3 "Frame sink" and §4 "Implementation": the tokens of the first frame
  chunk stay in every layer's KV cache for good and are concatenated to the
  keys and values of every attention; the rest of the cache is a short rolling
  window whose oldest frames are evicted as new ones arrive.
* §3.3 "Consistency between training and inference": W counts the preceding
  context frames; S sink frames are kept and never evicted; the resident KV is
  O(W + S) per layer (plus the frames being generated).
* §3.1 "KV recache": at a prompt switch, the cached K/V of the frames already
  generated are recomputed (with the new prompt) before generation goes on;
  §3.3 says the recache rebuilds the cache from the most recent frames.
* §4.4 (Table 4) "no KV cache" strategy: clear the whole cache at a switch.

Readings taken where the pages are silent:

* W counts preceding frames only; the chunk being generated is always visible
  in full to itself (chunk-level block causality).
* Softmax scale 1/sqrt(d); no positional term (q and k arrive pre-rotated).
* The window never duplicates a sink frame: window frames are those f >= S
  among the last W frames.
* Frame f < S lives in slot f; frame f >= S lives in ring slot
  S + ((f - S) mod W).  This is the canonical frame-to-slot map the cache
  state is compared against.
* Recache rewrites all R resident frames (sink frames ascending, then window
  frames ascending) in place; frame indices and the committed count are
  unchanged.  The optional prefill attention of a recache is block-causal over
  that list in blocks of C frames.

Two other readings are kept as options, because the pages leave them open:

* ``chunk_mask="frame"``: the model is called frame-level autoregressive, so a
  query of chunk frame t0 + i may instead see only the chunk's frames t0 .. t0 + i
  (plus every cached frame); the recache prefill then uses blocks of one frame.
* ``recache_scope="window"``: §3.3 says the recache rebuilds the cache only from
  the most recent W frames, so the sink may instead keep its K/V; only the window
  frames are rewritten, and the prefill queries of the window frames see the
  (unchanged) sink plus the fresh window, block-causal over the window.

Parity pins: every function here is pinned by tests under ``tests/`` that do
not call back into this module's own formulas (brute force, closed forms,
library routines, invariants, hand-written golden tables).
"""

from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# Frame bookkeeping (§3.3 "Frame sink"; §3.3 "Short window attention")
# ---------------------------------------------------------------------------


def sink_frames(S: int, n: int) -> list[int]:
    """Frames kept as the sink after n frames were committed: 0 .. min(S, n) - 1.

    §3.3 "Frame sink": the first frame chunk is pinned in the cache forever.
    """
    return list(range(min(S, n)))


def window_frames(S: int, W: int, n: int) -> list[int]:
    """The rolling window after n commits: the last W frames that are not sink frames.

    §3.3 "Short window attention" (fixed window of recent frames) and
    "Frame sink" (the rest of the cache rolls and evicts the oldest frames).
    """
    lo = max(S, n - W)
    return list(range(lo, n)) if n > lo else []


def resident_frames(S: int, W: int, n: int) -> list[int]:
    """All frames in a layer's cache after n commits, in logical order: sink asc, window asc."""
    return sink_frames(S, n) + window_frames(S, W, n)


def slot_of_frame(S: int, W: int, f: int) -> int:
    """Canonical physical slot of frame f: sink frames first, then a ring of W slots."""
    if f < S:
        return f
    if W <= 0:
        raise ValueError("frame %d cannot be resident when W = 0" % f)
    return S + (f - S) % W


def frame_of_slot(S: int, W: int, n: int) -> list[int]:
    """Expected slot table (length S + W) after n commits; -1 marks an empty slot."""
    table = [-1] * (S + W)
    for f in resident_frames(S, W, n):
        table[slot_of_frame(S, W, f)] = f
    return table


def visible_frames(S: int, W: int, C: int, t0: int) -> list[int]:
    """Frames one chunk starting at frame t0 attends to, in list order.

    §3.3 "Frame sink": the sink tokens are concatenated to the keys and values of
    every attention; "Short window attention": plus the recent window; the chunk
    itself is the last part of the list.
    """
    return sink_frames(S, t0) + window_frames(S, W, t0) + list(range(t0, t0 + C))


# ---------------------------------------------------------------------------
# Attention (explicit masked softmax over an explicit K/V list)
# ---------------------------------------------------------------------------


def masked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                     visible=None, rows=None, block_rows: int = 512) -> np.ndarray:
    """softmax(q k^T / sqrt(d)) v per head, in float64, with an optional key mask.

    q: [Lq, H, d]; k, v: [Lkv, H, d]; visible: None (every key visible) or a
    callable ``visible(qi) -> bool[Lkv]`` giving the keys query row qi may see.
    rows: optional array of query-row indices to evaluate (default: all).
    Returns [len(rows), H, d] float64.  The score matrix is materialised per
    block of query rows; nothing else is fused or reordered.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Lq, H, d = q.shape
    if rows is None:
        rows = np.arange(Lq)
    rows = np.asarray(rows, dtype=np.int64)
    scale = 1.0 / math.sqrt(d)
    out = np.empty((rows.shape[0], H, d), dtype=np.float64)
    kh = np.ascontiguousarray(k.transpose(1, 0, 2))  # [H, Lkv, d]
    vh = np.ascontiguousarray(v.transpose(1, 0, 2))
    for b0 in range(0, rows.shape[0], block_rows):
        r = rows[b0:b0 + block_rows]
        qh = q[r].transpose(1, 0, 2)  # [H, nr, d]
        scores = np.matmul(qh, kh.transpose(0, 2, 1)) * scale  # [H, nr, Lkv]
        if visible is not None:
            mask = np.stack([visible(int(i)) for i in r])  # [nr, Lkv]
            scores = np.where(mask[None, :, :], scores, -np.inf)
        scores = scores - scores.max(axis=2, keepdims=True)
        p = np.exp(scores)
        p = p / p.sum(axis=2, keepdims=True)
        out[b0:b0 + r.shape[0]] = np.matmul(p, vh).transpose(1, 0, 2)
    return out


def block_causal_visible(T: int, C: int, Lkv: int):
    """Key mask of the recache prefill: list blocks of C frames, block g sees blocks <= g.

    §3.1 "KV recache" re-encodes the generated frames as visual context the way
    they were generated: chunk by chunk, each chunk seeing itself and earlier ones.
    """
    block_tokens = C * T
    key_block = np.arange(Lkv) // block_tokens

    def visible(qi: int) -> np.ndarray:
        return key_block <= (qi // block_tokens)

    return visible


def prefix_then_block_causal_visible(n_prefix: int, block_tokens: int, Lkv: int):
    """Key mask with a fully visible prefix, then block causality over the rest.

    Keys [0, n_prefix) (cached frames) are seen by every query; key j >= n_prefix
    is seen by query row qi iff (j - n_prefix) // block_tokens <= qi // block_tokens.
    With one-frame blocks this is the frame-causal chunk of the "frame-level
    autoregressive" reading; with C-frame blocks after a sink prefix it is the
    keep-sink recache prefill.
    """
    kj = np.arange(Lkv)
    after = kj >= n_prefix
    key_block = np.where(after, (kj - n_prefix) // block_tokens, -1)

    def visible(qi: int) -> np.ndarray:
        return ~after | (key_block <= (qi // block_tokens))

    return visible


# ---------------------------------------------------------------------------
# The cache (one per layer) and the calls of the hot path
# ---------------------------------------------------------------------------


class OracleLayer:
    """One layer's KV cache as a dict frame -> (K_f, V_f), each [T, H, d] float64."""

    def __init__(self):
        self.n = 0
        self.frames: dict[int, tuple[np.ndarray, np.ndarray]] = {}


class OracleCache:
    """Per-layer rolling KV cache with a frame sink, kept as explicit frame lists."""

    def __init__(self, layers: int, heads: int, head_dim: int, tokens_per_frame: int,
                 sink_frames: int, window_frames: int, chunk_frames: int,
                 chunk_mask: str = "chunk", recache_scope: str = "resident"):
        if min(layers, heads, head_dim, tokens_per_frame, chunk_frames) < 1:
            raise ValueError("layers, heads, head_dim, tokens_per_frame, chunk_frames must be >= 1")
        if sink_frames < 0 or window_frames < 0:
            raise ValueError("sink_frames and window_frames must be >= 0")
        self.L, self.H, self.d = layers, heads, head_dim
        self.T, self.S, self.W, self.C = tokens_per_frame, sink_frames, window_frames, chunk_frames
        self.layers = [OracleLayer() for _ in range(layers)]
        self.set_chunk_mask(chunk_mask)
        self.set_recache_scope(recache_scope)

    def set_chunk_mask(self, mode: str) -> None:
        """"chunk" (default): a chunk sees all of its frames; "frame": only its frames up to the query's."""
        if mode not in ("chunk", "frame"):
            raise ValueError(mode)
        self.chunk_mask = mode

    def set_recache_scope(self, scope: str) -> None:
        """"resident" (default): recache rewrites sink and window; "window": the sink keeps its K/V."""
        if scope not in ("resident", "window"):
            raise ValueError(scope)
        self.recache_scope = scope

    def _block_frames(self) -> int:
        """Frames per causal block of the chunk / prefill masks."""
        return 1 if self.chunk_mask == "frame" else self.C

    # -- state ---------------------------------------------------------------
    def state(self, layer: int) -> tuple[int, list[int]]:
        """(frames committed, frame_of_slot table) of one layer."""
        lay = self.layers[layer]
        return lay.n, frame_of_slot(self.S, self.W, lay.n)

    def resident(self, layer: int) -> list[int]:
        return resident_frames(self.S, self.W, self.layers[layer].n)

    def frame_kv(self, layer: int, f: int) -> tuple[np.ndarray, np.ndarray]:
        return self.layers[layer].frames[f]

    # -- calls ---------------------------------------------------------------
    def attend(self, layer: int, q, k, v, commit: bool, rows=None) -> np.ndarray:
        """One query pass of the chunk that starts at frame t0 = frames committed.

        §3.3: keys/values = concat(sink frames, window frames, the chunk's own
        frames); every query of the chunk sees the whole list.  With commit,
        the chunk's K/V enter the cache afterwards and frames that fall out of
        the window are deleted (§3.3 "Frame sink": the rest of the cache is a
        rolling window with FIFO eviction).
        """
        lay = self.layers[layer]
        T, C = self.T, self.C
        q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
        assert q.shape == (C * T, self.H, self.d) and k.shape == q.shape and v.shape == q.shape
        t0 = lay.n
        past = resident_frames(self.S, self.W, t0)
        K = np.concatenate([lay.frames[f][0] for f in past] + [k], axis=0)
        V = np.concatenate([lay.frames[f][1] for f in past] + [v], axis=0)
        visible = None
        if self.chunk_mask == "frame":
            visible = prefix_then_block_causal_visible(len(past) * T, T, K.shape[0])
        out = masked_attention(q, K, V, visible=visible, rows=rows)
        if commit:
            self._commit(layer, k, v)
        return out

    def commit(self, layer: int, k, v) -> None:
        """The state change of a committing pass, for passes whose outputs nobody reads.

        Frames are kept as views of the given arrays (converted to float64);
        callers must not modify them afterwards.
        """
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        assert k.shape == (self.C * self.T, self.H, self.d) and v.shape == k.shape
        self._commit(layer, k, v)

    def _commit(self, layer: int, k: np.ndarray, v: np.ndarray) -> None:
        lay = self.layers[layer]
        T = self.T
        t0 = lay.n
        for i in range(self.C):
            f = t0 + i
            lay.frames[f] = (k[i * T:(i + 1) * T], v[i * T:(i + 1) * T])
        lay.n = t0 + self.C
        keep = set(resident_frames(self.S, self.W, lay.n))
        for f in list(lay.frames):
            if f not in keep:
                del lay.frames[f]

    def recache_frames(self, layer: int) -> list[int]:
        """Frames a recache rewrites, in the order of k_win / v_win."""
        n = self.layers[layer].n
        if self.recache_scope == "window":
            return window_frames(self.S, self.W, n)
        return resident_frames(self.S, self.W, n)

    def recache(self, layer: int, k_win, v_win) -> None:
        """§3.1 "KV recache": replace the K/V of the recached frames in list order.

        k_win, v_win: [R*T, H, d] for frames [sink asc, window asc] (scope
        "resident") or [window asc] (scope "window").  Frame indices and the
        committed count do not change.
        """
        lay = self.layers[layer]
        frames = self.recache_frames(layer)
        if not frames:
            raise ValueError("recache of an empty layer")
        T = self.T
        k_win = np.asarray(k_win, dtype=np.float64)
        v_win = np.asarray(v_win, dtype=np.float64)
        assert k_win.shape == (len(frames) * T, self.H, self.d) and v_win.shape == k_win.shape
        for i, f in enumerate(frames):
            lay.frames[f] = (k_win[i * T:(i + 1) * T], v_win[i * T:(i + 1) * T])

    def recache_attend(self, layer: int, q_win, k_win, v_win, rows=None) -> np.ndarray:
        """Recache with the prefill attention: block-causal over the recached list.

        Scope "resident": the list [sink asc, window asc] is cut into blocks of C
        frames (one frame with the frame mask); query rows in block g see key
        blocks 0..g.  Scope "window": the queries are the window frames'; they
        see every sink frame (its cached K/V) plus the fresh window, block-causal
        over the window.  The fresh K/V then replace the recached frames as in
        :meth:`recache`.
        """
        lay = self.layers[layer]
        R = len(self.recache_frames(layer))
        if R == 0:
            raise ValueError("recache of an empty layer")
        q_win = np.asarray(q_win, dtype=np.float64)
        k_win = np.asarray(k_win, dtype=np.float64)
        v_win = np.asarray(v_win, dtype=np.float64)
        T = self.T
        L = R * T
        assert q_win.shape == (L, self.H, self.d)
        block = self._block_frames() * T
        if self.recache_scope == "window":
            sink = sink_frames(self.S, lay.n)
            K = np.concatenate([lay.frames[f][0] for f in sink] + [k_win], axis=0)
            V = np.concatenate([lay.frames[f][1] for f in sink] + [v_win], axis=0)
            visible = prefix_then_block_causal_visible(len(sink) * T, block, K.shape[0])
            out = masked_attention(q_win, K, V, visible=visible, rows=rows)
        else:
            out = masked_attention(q_win, k_win, v_win, visible=block_causal_visible(block, 1, L), rows=rows)
        self.recache(layer, k_win, v_win)
        return out

    def reset(self) -> None:
        """§4.4 Table 4, "no KV cache": clear every layer."""
        for lay in self.layers:
            lay.n = 0
            lay.frames.clear()

    # -- expected raw cache contents -----------------------------------------
    def expected_slots(self, layer: int) -> dict[int, int]:
        """slot -> frame for every occupied slot (what the raw cache must hold)."""
        n, table = self.state(layer)
        return {s: f for s, f in enumerate(table) if f >= 0}


def lkv_tokens(S: int, W: int, C: int, T: int, t0: int) -> int:
    """Length of the attended K/V list of the chunk at t0, in tokens."""
    return len(visible_frames(S, W, C, t0)) * T


def attention_flops(Lq: int, Lkv: int, H: int, d: int) -> float:
    """Algorithmic flops of one attend: QK^T and PV, 2 flops per multiply-add each."""
    return 4.0 * Lq * Lkv * H * d
