"""bench.py's work accounting against the oracle's definitions (CPU).

The reported TFLOP/s count only the query-key pairs a query may see, and the
append bandwidth counts only the frames a commit keeps.  These tests recount both
from the oracle's own visibility masks and commit bookkeeping, for the default
reading and for the two options.
"""

import os
import sys

import numpy as np
import pytest

from oracle import ll_oracle as O
from tests.conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402
import llsynth  # noqa: E402


def mask_pairs(visible, Lq):
    return int(sum(int(np.count_nonzero(visible(i))) for i in range(Lq)))


SHAPES = [llsynth.Shape(1, 1, 1, 4, 3, 6, 3), llsynth.Shape(1, 1, 1, 5, 0, 4, 2), llsynth.Shape(1, 1, 1, 3, 2, 0, 3),
          llsynth.Shape(1, 1, 1, 2, 1, 2, 1)]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s)[5:] for s in SHAPES])
def test_chunk_pairs_match_the_oracle_masks(shape):
    T, S, W, C = shape.tokens_per_frame, shape.sink_frames, shape.window_frames, shape.chunk_frames
    L = C * T
    for t0 in range(0, 8 * C, C):
        assert bench.resident_count(S, W, t0) == len(O.resident_frames(S, W, t0))
        past = len(O.resident_frames(S, W, t0)) * T
        assert bench.chunk_pairs(shape, t0, "chunk") == L * O.lkv_tokens(S, W, C, T, t0)
        frame_visible = O.prefix_then_block_causal_visible(past, T, past + L)
        assert bench.chunk_pairs(shape, t0, "frame") == mask_pairs(frame_visible, L)


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s)[5:] for s in SHAPES])
def test_prefill_pairs_match_the_oracle_masks(shape):
    T, S, W, C = shape.tokens_per_frame, shape.sink_frames, shape.window_frames, shape.chunk_frames
    for n in range(C, 8 * C, C):
        for mask in ("chunk", "frame"):
            block = (1 if mask == "frame" else C) * T
            R = len(O.resident_frames(S, W, n)) * T
            want = mask_pairs(O.block_causal_visible(block, 1, R), R)
            assert bench.prefill_pairs(shape, n, mask, "resident") == want
            sink = min(S, n) * T
            win = len(O.window_frames(S, W, n)) * T
            want = mask_pairs(O.prefix_then_block_causal_visible(sink, block, sink + win), win) if win else 0
            assert bench.prefill_pairs(shape, n, mask, "window") == want


def test_frames_written_match_the_oracle_commit():
    for S, W, C in [(3, 9, 3), (4, 2, 3), (0, 6, 3), (2, 0, 3), (3, 1, 4)]:
        shape = llsynth.Shape(1, 1, 1, 1, S, W, C)
        c = O.OracleCache(1, 1, 1, 1, S, W, C)
        z = np.zeros((C, 1, 1))
        for _ in range(8):
            t0 = c.state(0)[0]
            c.commit(0, z, z)
            kept = [f for f in O.resident_frames(S, W, t0 + C) if f >= t0]
            assert bench.frames_written(shape, t0) == len(kept), (S, W, C, t0)


def test_stream_plan_matches_visible_frames():
    s = llsynth.STREAM30
    plan = bench.stream_plan(s, llsynth.STREAM30_CHUNKS)
    for c, (t0, lkv) in enumerate(plan):
        assert t0 == c * s.chunk_frames
        assert lkv == O.lkv_tokens(s.sink_frames, s.window_frames, s.chunk_frames, s.tokens_per_frame, t0)
    # steady state: 0.6728 TFLOP per attend launch of the Wan-shaped layer
    flops = bench.pair_flops(bench.chunk_pairs(s, 12, "chunk"), s.heads, s.head_dim)
    assert abs(flops - 0.672841728e12) < 1.0


def test_code_hash_ignores_comments_only():
    """The traffic record is keyed by a hash of the kernel's code: comment and blank-line
    edits keep it, any change to the code changes it."""
    src = "int f(int x) {  // doubles x\n  return 2 * x;\n}\n"
    base = bench.code_hash([src, "#define N 4\n"])
    assert bench.code_hash(["// header\n\n" + src.replace("doubles x", "twice x") + "\n\n",
                            "#define N 4  // four\n"]) == base
    assert bench.code_hash([src.replace("2 * x", "3 * x"), "#define N 4\n"]) != base
    assert bench.code_hash([src, "#define N 5\n"]) != base
    # file boundaries count: moving a line from one file to the next changes the hash
    assert bench.code_hash([src + "#define N 4\n", ""]) != base


def test_traffic_record_names_a_code_hash():
    rec = {}
    with open(os.path.join(ROOT, "profiles", "attend_tc_traffic.txt")) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                rec[k.strip()] = v.strip()
    assert len(rec["source_hash"]) == 16 and int(rec["source_hash"], 16) >= 0
    assert float(rec["dram_bytes_per_launch"]) > float(rec["algorithmic_bytes_per_launch"]) > 0
