"""ll_attend_chunk_noalloc through the C ABI: against ll_attend_chunk and the oracle.

ll_attend_chunk_noalloc is the chunk attention for callers that may not
allocate device memory: a host program whose memory manager owns the GPU's
whole budget, a plugin interface that forbids its libraries to allocate, or a
real-time loop that cannot absorb the host blocking and device synchronisation
of cudaMalloc / cudaFree.  It runs the same tensor-core kernel with the scratch
for its split work items in a static device array of the library instead of
memory allocated with the cache, so its outputs must equal ll_attend_chunk's
bit for bit, and sampled rows must match the float64 oracle ("LongLive", §3.3
"Frame sink" + "Short window attention": the chunk attends to the resident
sink and window frames and to itself) within max |err| <= 1e-2 and relative
L2 <= 5e-3.

The file name puts it last in collection order, so a run that stops at the
first failure has run every other test before this one.
"""

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


def _resident_rows(ll, cache, layer):
    """One layer's K and V cache as device tensors [H, (S+W)*T, d]; resident frames fill the first rows."""
    hk, hv = ll.ll_cache_read(cache, layer)
    H, slots, T, d = hk.shape
    return hk.reshape(H, slots * T, d).cuda(), hv.reshape(H, slots * T, d).cuda()


def test_noalloc_matches_attend_chunk_and_oracle_on_two_calls(ll):
    s = llsynth.SINGLE_LAYER  # 12 heads x 128, 1560 tokens per frame, chunks of 3, sink 3, window 9
    H, d, T, S, W, C = s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames, s.chunk_frames
    L = C * T
    rows = sample_rows(L, 160, seed=3)
    # Two cache states with different schedules: sink + full window (184 key tiles per
    # work item) and sink only (74); both split their left-over items across CTAs.
    cases = []
    for name, chunks in (("sink+window", 4), ("sink only", 1)):
        st = Lockstep(ll, 1, H, d, T, S, W, C, torch.bfloat16, keep_frames=False)
        for c in range(chunks):
            q, k, v = (llsynth.seeded_normal(("noalloc-fill", name, c, t), (L, H, d), device="cuda") for t in "qkv")
            st.attend(0, q, k, v, commit=True, check=False)
        n, _ = ll.ll_cache_state(st.cache, 0)
        R = ll.ll_resident_count(S, W, n)
        assert R == min(S, n) + min(W, max(0, n - S))
        q, k, v = (llsynth.seeded_normal(("noalloc", name, t), (L, H, d), device="cuda") for t in "qkv")
        ref = torch.empty_like(q)
        ll.ll_attend_chunk(st.cache, 0, q, k, v, ref, False)
        want = st.orc.attend(0, f64(q), f64(k), f64(v), False, rows=rows)
        kc, vc = _resident_rows(ll, st.cache, 0)
        cases.append((name, q, k, v, kc, vc, R * T, ref, want))
        st.close()

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.full_like(case[1], float("nan")) for case in cases]
    torch.cuda.synchronize()
    free_before_second = None
    for i, (name, q, k, v, kc, vc, La, _, _) in enumerate(cases):
        if i == 1:
            torch.cuda.synchronize()
            free_before_second = torch.cuda.mem_get_info()[0]
        ll.ll_attend_chunk_noalloc(q, kc, vc, La, k, v, outs[i], err_word=err)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before_second, "the second call changed free device memory"
    assert int(err.item()) == 0
    for (name, *_, ref, want), out in zip(cases, outs):
        # same kernel, same schedule, same inputs: the same bits as ll_attend_chunk
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), name
        compare(out[torch.as_tensor(rows, device="cuda")], want, "noalloc vs oracle, %s" % name)


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
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    orc = oracle.OracleCache(1, H, d, L, 0, 0, 1)
    compare(out, orc.attend(0, f64(q), f64(k), f64(v), False), "noalloc without cached rows vs oracle")

    q96 = torch.zeros((8, 1, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ll.LLError) as e:
        ll.ll_attend_chunk_noalloc(q96, None, None, 0, q96.clone(), q96.clone(), q96.clone())
    assert e.value.status == ll.LL_ERR_UNSUPPORTED
    with pytest.raises(ll.LLError) as e:
        ll.ll_attend_chunk_noalloc(q, None, None, 0, k, v, q)  # out aliases q
    assert e.value.status == ll.LL_ERR_INVALID_ARG
    with pytest.raises(ValueError):  # an error word needs room for one int32
        ll.ll_attend_chunk_noalloc(q, None, None, 0, k, v, out, err_word=torch.zeros(0, dtype=torch.int32,
                                                                                      device="cuda"))
