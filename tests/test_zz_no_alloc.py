"""ll_attend_chunk_noalloc against ll_attend_chunk, through the C ABI.

ll_attend_chunk_noalloc is the chunk attention for callers that may not
allocate device memory: a host program whose memory manager owns the GPU's
whole budget, a plugin interface that forbids its libraries to allocate, or a
real-time loop that cannot absorb the host blocking and device synchronisation
of cudaMalloc / cudaFree.  It runs the same tensor-core kernel with the scratch
for its split work items in a static device array of the library instead of
memory allocated with the cache.

The file name puts it last in collection order, so a run that stops at the
first failure has run every other test before this one.
"""

import pytest
import torch

import llsynth
from tests.gpu_util import compare, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    torch.cuda.set_device(0)
    return mod


def _resident_rows(ll, cache, layer):
    """One layer's K and V cache as device tensors [H, (S+W)*T, d]; resident frames fill the first rows."""
    hk, hv = ll.ll_cache_read(cache, layer)
    H, slots, T, d = hk.shape
    return hk.reshape(H, slots * T, d).cuda(), hv.reshape(H, slots * T, d).cuda()


def test_noalloc_matches_attend_chunk_on_two_calls(ll):
    s = llsynth.SINGLE_LAYER  # 12 heads x 128, 1560 tokens per frame, chunks of 3, sink 3, window 9
    H, d, T, S, W, C = s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames, s.chunk_frames
    L = C * T
    # Two cache states with different schedules: sink + full window (184 key tiles per
    # work item) and sink only (74); both split their left-over items across CTAs.
    cases = []
    for name, chunks in (("sink+window", 4), ("sink only", 1)):
        cache = ll.ll_cache_create(1, H, d, T, S, W, C, ll.LL_BF16)
        for c in range(chunks):
            q, k, v = (llsynth.seeded_normal(("noalloc-fill", name, c, t), (L, H, d), device="cuda") for t in "qkv")
            ll.ll_attend_chunk(cache, 0, q, k, v, torch.empty_like(q), True)
        n, _ = ll.ll_cache_state(cache, 0)
        R = ll.ll_resident_count(S, W, n)
        assert R == min(S, n) + min(W, max(0, n - S))
        q, k, v = (llsynth.seeded_normal(("noalloc", name, t), (L, H, d), device="cuda") for t in "qkv")
        ref = torch.empty_like(q)
        ll.ll_attend_chunk(cache, 0, q, k, v, ref, False)
        kc, vc = _resident_rows(ll, cache, 0)
        cases.append((name, q, k, v, kc, vc, R * T, ref))
        cache.close()

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.full_like(case[1], float("nan")) for case in cases]
    torch.cuda.synchronize()
    free_before_second = None
    for i, (name, q, k, v, kc, vc, La, _) in enumerate(cases):
        if i == 1:
            torch.cuda.synchronize()
            free_before_second = torch.cuda.mem_get_info()[0]
        ll.ll_attend_chunk_noalloc(q, kc, vc, La, k, v, outs[i], err_word=err)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before_second, "the second call changed free device memory"
    assert int(err.item()) == 0
    for (name, *_, ref), out in zip(cases, outs):
        compare(out, f64(ref), "noalloc vs ll_attend_chunk, %s" % name)


def test_noalloc_without_cached_rows_and_bad_requests(ll):
    H, d, L = 3, 64, 300
    q, k, v = (llsynth.seeded_normal(("noalloc-empty", t), (L, H, d), device="cuda") for t in "qkv")
    out = torch.full_like(q, float("nan"))
    ll.ll_attend_chunk_noalloc(q, None, None, 0, k, v, out)
    cache = ll.ll_cache_create(1, H, d, L, 0, 0, 1, ll.LL_BF16)  # no sink, no window: attention within the chunk
    ref = torch.empty_like(q)
    ll.ll_attend_chunk(cache, 0, q, k, v, ref, False)
    torch.cuda.synchronize()
    cache.close()
    compare(out, f64(ref), "noalloc without cached rows")

    q96 = torch.zeros((8, 1, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ll.LLError) as e:
        ll.ll_attend_chunk_noalloc(q96, None, None, 0, q96.clone(), q96.clone(), q96.clone())
    assert e.value.status == ll.LL_ERR_UNSUPPORTED
    with pytest.raises(ll.LLError) as e:
        ll.ll_attend_chunk_noalloc(q, None, None, 0, k, v, q)  # out aliases q
    assert e.value.status == ll.LL_ERR_INVALID_ARG
