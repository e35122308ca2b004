"""A stream of ll_attend_chunk calls recorded as one CUDA graph replays the same work.

The library keeps its frame bookkeeping on the host and enqueues plain kernel
launches, so a whole stream step from an empty cache (every layer, every chunk,
each pass committing) can be recorded with torch.cuda.graph and replayed
("LongLive", §3.3 "Short window attention": the chunk-by-chunk streaming loop
over the rolling sink + window cache).  The replay's outputs and raw cache bytes
must equal an eager run's bit for bit, and the replayed outputs must match the
float64 oracle driven through the same calls (sampled query rows, every layer
and chunk, the usual bound: max |err| <= 1e-2, relative L2 <= 5e-3).  The e4m3
key-and-value cache records its rounding kernel in the graph as well; its oracle
is fed the rounded q, k and v.
"""

import pytest
import torch

import llsynth
import oracle
from tests.gpu_util import compare, f64, round_e4m3, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    torch.cuda.set_device(0)
    return mod


@pytest.mark.parametrize("mask,kind", [("chunk", "bf16"), ("frame", "bf16"), ("chunk", "fp8")])
def test_stream_replayed_from_a_cuda_graph_equals_eager_and_oracle(ll, mask, kind):
    layers, H, D, T, S, W, C, chunks = 2, 12, 128, 1040, 3, 6, 3, 6  # 156 items: split tail too
    L = C * T
    cache = ll.ll_cache_create(layers, H, D, T, S, W, C, ll.LL_FP8 if kind == "fp8" else ll.LL_BF16)
    ll.ll_set_chunk_mask(cache, mask)
    inputs = [[tuple(llsynth.seeded_normal(("graph", l, c, t), (L, H, D), device="cuda") for t in "qkv")
               for c in range(chunks)] for l in range(layers)]
    outs = [[torch.empty((L, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(chunks)]
            for _ in range(layers)]

    def step():
        ll.ll_reset(cache)
        st = torch.cuda.current_stream()
        for c in range(chunks):
            for l in range(layers):
                ll.ll_attend_chunk(cache, l, *inputs[l][c], outs[l][c], True, st)

    step()
    torch.cuda.synchronize()
    eager = [[o.clone() for o in row] for row in outs]
    eager_raw = [ll.ll_cache_read(cache, l) for l in range(layers)]
    for row in outs:
        for o in row:
            o.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):  # replay twice: the second replay starts from the first one's cache
        g.replay()
        torch.cuda.synchronize()
        for l in range(layers):
            for c in range(chunks):
                assert torch.equal(outs[l][c], eager[l][c]), (l, c)
            k, v = ll.ll_cache_read(cache, l)
            assert torch.equal(k, eager_raw[l][0]) and torch.equal(v, eager_raw[l][1]), l

    # the replayed outputs against the oracle fed the same calls in the same order
    orc = oracle.OracleCache(layers, H, D, T, S, W, C)
    orc.set_chunk_mask(mask)
    rows = sample_rows(L, 96, seed=7)
    for c in range(chunks):
        for l in range(layers):
            q, k, v = (f64(round_e4m3(t)) if kind == "fp8" else f64(t) for t in inputs[l][c])
            want = orc.attend(l, q, k, v, True, rows=rows)
            compare(outs[l][c][torch.as_tensor(rows, device="cuda")], want,
                    "graph replay vs oracle, %s cache, mask %s, layer %d chunk %d" % (kind, mask, l, c))
    for l in range(layers):
        assert ll.ll_cache_state(cache, l) == orc.state(l), l
    cache.close()
