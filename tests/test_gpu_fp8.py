"""The e4m3 caches through the C ABI, against the float64 oracle.

LL_BF16_K8 ("keys"): keys are stored in the K cache rounded to FP8 e4m3, and Q K^T
runs on the FP8 tensor-core path (tcgen05.mma kind::f8f6f4) with q and the fresh
keys rounded the same way; V, P and the outputs stay bf16.  LL_FP8 ("kv"): the
values are stored rounded to e4m3 as well, and P V runs on fp16 operands (V widened
exactly, P rounded to fp16).  ("LongLive", Abstract and §5 Conclusion: quantized
inference; §3.3 "Frame sink" + "Short window attention" for what the attention
computes.)  Rounding is a defined input step, so the oracle is fed the e4m3-rounded
q and k (and v for LL_FP8) and the usual bound holds: max |err| <= 1e-2, relative
L2 <= 5e-3.  Cache state bit-exact; the raw slots hold exactly the e4m3 bytes of the
committed keys (and values), or the committed bf16 values.
"""

import pytest
import torch

import llsynth
from tests.gpu_util import Lockstep, f64, round_e4m3, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    torch.cuda.set_device(0)
    return mod


SHAPES = [
    # H, T,   S, W, C
    (2, 40, 3, 6, 3),     # 120 queries: one item per head
    (3, 100, 3, 9, 3),    # 300 queries (ragged second item), cache tiles that end mid-tile
    (2, 130, 0, 4, 2),    # no sink, window wraps
    (64, 200, 2, 4, 3),   # 192 items: a whole round, then a split tail
]


KINDS = ["keys", "kv"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("mask", ["chunk", "frame"])
@pytest.mark.parametrize("shape", SHAPES, ids=["-".join(map(str, s)) for s in SHAPES])
def test_fp8_keys_stream_recache_and_prefill(ll, shape, mask, kind):
    H, T, S, W, C = shape
    D = 128
    st = Lockstep(ll, 2, H, D, T, S, W, C, torch.bfloat16, key_fp8=True, value_fp8=(kind == "kv"))
    st.set_options(chunk_mask=mask)
    L = C * T
    for c in range(6):
        for layer in (0, 1):
            q, k, v = (llsynth.seeded_normal(("fp8", shape, mask, layer, c, t), (L, H, D), device="cuda")
                       for t in "qkv")
            st.attend(layer, q, k, v, commit=True, what="fp8 %s %s %s L%d c%d" % (kind, shape, mask, layer, c))
        st.check_state()
    st.check_raw(0)
    st.check_raw(1)
    R = len(st.orc.recache_frames(1))
    if R:
        qw, kw, vw = (llsynth.seeded_normal(("fp8-rc", shape, mask, t), (R * T, H, D), device="cuda") for t in "qkv")
        st.recache_attend(1, qw, kw, vw, what="fp8 %s prefill %s %s" % (kind, shape, mask))
        kw2, vw2 = (llsynth.seeded_normal(("fp8-rc2", shape, mask, t), (R * T, H, D), device="cuda") for t in "kv")
        st.recache(0, kw2, vw2)
        st.check_state()
        st.check_raw(0)
        st.check_raw(1)
        for layer in (0, 1):
            q, k, v = (llsynth.seeded_normal(("fp8-after", shape, mask, layer, t), (L, H, D), device="cuda")
                       for t in "qkv")
            st.attend(layer, q, k, v, commit=False, what="fp8 %s after recache %s L%d" % (kind, shape, layer))
    st.close()


@pytest.mark.parametrize("kind", KINDS)
def test_fp8_keys_keep_sink_recache(ll, kind):
    H, D, T, S, W, C = 2, 128, 64, 3, 6, 3
    st = Lockstep(ll, 1, H, D, T, S, W, C, torch.bfloat16, key_fp8=True, value_fp8=(kind == "kv"))
    st.set_options(recache_scope="window")
    for c in range(4):
        q, k, v = (llsynth.seeded_normal(("fp8-ks", c, t), (C * T, H, D), device="cuda") for t in "qkv")
        st.attend(0, q, k, v, commit=True, what="fp8 keep-sink c%d" % c)
    R = len(st.orc.recache_frames(0))
    qw, kw, vw = (llsynth.seeded_normal(("fp8-ks-rc", t), (R * T, H, D), device="cuda") for t in "qkv")
    st.recache_attend(0, qw, kw, vw, what="fp8 keep-sink prefill")
    st.check_state()
    st.check_raw(0)
    st.close()


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fp8_keys_wan_layer(ll, out_dtype, kind):
    """The single Wan-shaped layer (per-head scales 0.5-2, 23400 keys), sampled rows."""
    s = llsynth.SINGLE_LAYER
    st = Lockstep(ll, 1, s.heads, s.head_dim, s.tokens_per_frame, s.sink_frames, s.window_frames, s.chunk_frames,
                  torch.bfloat16, key_fp8=True, value_fp8=(kind == "kv"))
    ll.ll_set_output_dtype(st.cache, out_dtype)
    if out_dtype == torch.bfloat16:
        st.atol = None  # the bf16 rounding of a value within 1e-2 of the oracle (see compare)
    for c in range(4):
        q, k, v = (llsynth.seeded_normal(("fp8-wan", c, t), (s.chunk_tokens, s.heads, s.head_dim), device="cuda",
                                         per_head_scale=True) for t in "qkv")
        st.attend(0, q, k, v, commit=True, check=False)
    rows = sample_rows(s.chunk_tokens, 256, seed=13)
    for p in range(2):
        q, k, v = (llsynth.seeded_normal(("fp8-wan-q", p, t), (s.chunk_tokens, s.heads, s.head_dim), device="cuda",
                                         per_head_scale=True) for t in "qkv")
        st.attend(0, q, k, v, commit=(p == 1), rows=rows, what="fp8 %s Wan layer pass %d" % (kind, p))
        st.check_state()
    st.check_raw(0)
    st.close()


@pytest.mark.parametrize("kind", KINDS)
def test_fp8_keys_round_like_the_reference_helper(ll, kind):
    """The library's e4m3 rounding of the committed keys (and values), byte for byte,
    including values beyond the format's range (saturated at +-448), ties and subnormals."""
    H, D, T = 1, 128, 8
    st = Lockstep(ll, 1, H, D, T, 1, 0, 1, torch.bfloat16, key_fp8=True, value_fp8=(kind == "kv"))
    ramp = torch.linspace(-600.0, 600.0, T * H * D).reshape(T, H, D)
    special = torch.tensor([2.0 ** -9, 3 * 2.0 ** -10, 2.0 ** -10, 0.0, -0.0, 1.0625, 1.1875, 240.0, 464.0, 447.0])
    ramp.view(-1)[:special.numel()] = special
    k = ramp.to(torch.bfloat16).cuda()
    v = k.flip(0) if kind == "kv" else torch.ones_like(k)
    st.attend(0, torch.zeros_like(k), k, v, commit=True, check=False)
    hk, hv = ll.ll_cache_read(st.cache, 0)
    assert torch.equal(hk[:, 0], round_e4m3(k).view(torch.uint8).permute(1, 0, 2))
    if kind == "kv":
        assert torch.equal(hv[:, 0], round_e4m3(v).view(torch.uint8).permute(1, 0, 2))
    else:
        assert torch.equal(hv[:, 0].view(torch.int16), v.cpu().view(torch.int16).permute(1, 0, 2))
    st.close()


@pytest.mark.parametrize("code", ["LL_BF16_K8", "LL_FP8"])
def test_fp8_keys_unsupported_head_dim(ll, code):
    with pytest.raises(ll.LLError) as e:
        ll.ll_cache_create(1, 2, 64, 16, 3, 6, 3, getattr(ll, code))
    assert e.value.status == ll.LL_ERR_UNSUPPORTED
