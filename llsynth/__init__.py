"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle's callers.

This module holds no attention or cache arithmetic: only workload shapes and
seeded random tensors.  Neither the CUDA library nor the oracle imports it;
the tests and ``bench.py`` draw inputs here and hand the same values to both.

Workloads (shapes of the Wan2.1-T2V-1.3B self-attention that LongLive builds
on: 832x480 video at 16 FPS -> a 30x52 latent patch grid = 1560 tokens per
latent frame, 12 heads of dimension 128, chunks of 3 latent frames, a sink of
the first chunk and a window of 9 frames -- "LongLive", §4 Implementation and
§3.3 / Figure 5 "window 9 + sink 3"):

* ``tiny``: 1 layer, H=2, d=64, T=16, C=3, S=3, W=6; 8 chunks x 2 passes,
  q/k/v i.i.d. N(0,1)/sqrt(64) from numpy seed 0; a recache before chunk 5
  with fresh N(0,1) K/V for the resident frames.
* ``single_layer``: H=12, d=128, T=1560, C=3, S=3, W=9; cache pre-filled so
  that 12 frames are resident (attended list = 15 frames = 23400 tokens);
  bf16 N(0,1) scaled per head by s_h = 0.5 + 1.5 h / (H - 1); 4 passes,
  commit on the last.
* ``stream30``: 30 layers x 20 chunks, one committed pass per chunk,
  independent seeded N(0,1) q/k/v per layer and chunk.
* ``recache30``: 30 layers x 40 chunks; before (0-based) chunks 10, 20 and 30
  every layer runs a recache prefill of its 12 resident frames with fresh
  seeded q/k/v.
* ``sweep``: 1 layer x 320 chunks for W in {3,6,9,12,18} x S in {0,3}.
"""

from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Shape:
    layers: int
    heads: int
    head_dim: int
    tokens_per_frame: int
    sink_frames: int
    window_frames: int
    chunk_frames: int

    @property
    def chunk_tokens(self) -> int:
        return self.chunk_frames * self.tokens_per_frame


TINY = Shape(layers=1, heads=2, head_dim=64, tokens_per_frame=16,
             sink_frames=3, window_frames=6, chunk_frames=3)
WAN = dict(heads=12, head_dim=128, tokens_per_frame=1560, chunk_frames=3)
SINGLE_LAYER = Shape(layers=1, sink_frames=3, window_frames=9, **WAN)
STREAM30 = Shape(layers=30, sink_frames=3, window_frames=9, **WAN)
RECACHE30 = STREAM30
SWEEP_W = (3, 6, 9, 12, 18)
SWEEP_S = (0, 3)

TINY_CHUNKS = 8
TINY_PASSES = 2
TINY_RECACHE_BEFORE_CHUNK = 5
SINGLE_LAYER_PASSES = 4
STREAM30_CHUNKS = 20
RECACHE30_CHUNKS = 40
RECACHE30_SWITCHES = (10, 20, 30)
SWEEP_CHUNKS = 320
SWEEP_CHECK_CHUNKS = (1, 2, 4, 80, 320)  # 1-based chunk numbers


def seed_of(*key) -> int:
    """A stable 63-bit seed from a tuple key (config, layer, chunk, pass, tensor)."""
    h = hashlib.sha256(repr(key).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def head_scale(heads: int) -> torch.Tensor:
    """Per-head input scale s_h = 0.5 + 1.5 h / (H - 1) (1.0 for a single head)."""
    if heads == 1:
        return torch.ones(1)
    return 0.5 + 1.5 * torch.arange(heads, dtype=torch.float64) / (heads - 1)


def seeded_normal(key, shape, dtype=torch.bfloat16, device="cpu", std=1.0,
                  per_head_scale: bool = False) -> torch.Tensor:
    """N(0, std^2) tensor of ``shape`` ([tokens, H, d]) drawn from the seed of ``key``.

    The draw is float32 then rounded to ``dtype`` (round to nearest even).  The
    same key on the same device type always gives the same bytes.
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed_of(*key))
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    if per_head_scale:
        s = head_scale(shape[1]).to(device=device, dtype=torch.float32)
        x = x * s.view(1, -1, 1)
    return x.to(dtype)


def tiny_inputs(dtype=torch.float32, recache_frames: int = 9):
    """The tiny workload's tensors, drawn from numpy ``default_rng(0)`` in a fixed order.

    Returns dict with ``passes[c][p] = (q, k, v)`` for chunk c and pass p, each
    [48, 2, 64], i.i.d. N(0,1)/sqrt(64); ``recache_kv = (k_win, v_win)`` of
    fresh N(0,1) values for the ``recache_frames`` frames resident before
    chunk 5 (the caller states how many: 3 sink + 6 window frames = 9); and
    ``recache_q`` (N(0,1)/sqrt(64)) for the prefill variant.  All are CPU
    tensors of ``dtype``.
    """
    s = TINY
    rng = np.random.default_rng(0)
    L = s.chunk_tokens
    shp = (L, s.heads, s.head_dim)
    scale = 1.0 / np.sqrt(s.head_dim)

    def draw(shape, mult):
        return torch.from_numpy(rng.standard_normal(shape) * mult).to(dtype)

    passes = []
    for _c in range(TINY_CHUNKS):
        row = []
        for _p in range(TINY_PASSES):
            row.append(tuple(draw(shp, scale) for _ in range(3)))
        passes.append(row)
    r_frames = recache_frames
    wshape = (r_frames * s.tokens_per_frame, s.heads, s.head_dim)
    k_win = draw(wshape, 1.0)
    v_win = draw(wshape, 1.0)
    q_win = draw(wshape, scale)
    return {"passes": passes, "recache_kv": (k_win, v_win), "recache_q": q_win,
            "recache_frames": r_frames}
