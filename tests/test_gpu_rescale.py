"""Rows whose max score jumps after the first key tile: the reference-max moves.

The attention kernels keep a reference max per query row and move it (and
rescale O and the row sum) only when a tile's max grows more than 2^8 past it.  With ordinary inputs that
never happens after the first tile, so these inputs force it: every query points
along one direction u, the first key tile holds small noise, and single keys
along u with growing length (scores about 18, 43 and 64 above the first tile's
max, in log2 units, at head_dim 128) sit in the low half of one later tile, in
the high half of another and in the chunk's own keys.  Every row's softmax is then
dominated by keys the first tile did not see, in both halves of a tile, and the
outputs must still match the float64 oracle ("LongLive", §3.3: softmax over
[sink || window || chunk]) within max |err| <= 1e-2 and relative L2 <= 5e-3.
"""

import pytest
import torch

import llsynth
from tests.gpu_util import Lockstep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    torch.cuda.set_device(0)
    return mod


def direction(D):
    u = llsynth.seeded_normal(("direction", D), (D,)).float()
    return u / u.norm()


def spiky(tag, rows, H, D, spikes, scale, plus=0.0, dtype=torch.bfloat16):
    """Small N(0,1) * 0.05 rows (plus `plus` * u) with row i replaced by scale[i] * u, where u
    is a fixed unit direction; `dtype` (bf16) on the GPU."""
    u = direction(D)
    x = llsynth.seeded_normal((tag, "noise"), (rows, H, D)).float() * 0.05 + plus * u
    for r, c in zip(spikes, scale):
        x[r] = c * u
    return x.to(dtype).cuda()


KERNELS = ["one_cta", "pair", "fp8_keys", "fp8_kv", "one_cta_d64", "tf32_d64"]


@pytest.mark.parametrize("kernel", KERNELS)
def test_reference_max_moves_after_the_first_tile(ll, kernel):
    """one_cta / pair: bf16 at head_dim 128 on the one-CTA and CTA-pair kernels; fp8_keys /
    fp8_kv: the e4m3 caches; one_cta_d64: bf16 at head_dim 64; tf32_d64: fp32 at head_dim 64
    (tf32 operands)."""
    D = 64 if kernel.endswith("_d64") else 128
    dt = torch.float32 if kernel == "tf32_d64" else torch.bfloat16
    H, T, S, W, C = 2, 64, 2, 6, 2  # a 128-key tile = 2 frames; 8 resident frames = 4 cache tiles
    st = Lockstep(ll, 1, H, D, T, S, W, C, dt, key_fp8=(kernel == "fp8_keys"), value_fp8=(kernel == "fp8_kv"))
    ll.ll_debug_pair_kernel(st.cache, kernel == "pair")
    L = C * T
    # frames 0..7 resident in slots 0..7 after four commits; spikes along u: frame 2 token 5
    # (keys 0-63 of cache tile 1) and frame 5 token 7 (keys 64-127 of cache tile 2)
    for c in range(4):
        spikes, scale = [], []
        if c == 1:
            spikes, scale = [5], [10.0]           # frame 2, token 5
        if c == 2:
            spikes, scale = [T + 7], [24.0]       # frame 5, token 7
        k = spiky(("rescale-k", D, c), L, H, D, spikes, scale, dtype=dt)
        v = llsynth.seeded_normal(("rescale-v", D, c), (L, H, D), dtype=dt, device="cuda")
        q = llsynth.seeded_normal(("rescale-qf", D, c), (L, H, D), dtype=dt, device="cuda")
        st.attend(0, q, k, v, commit=True, check=False)
    assert st.orc.resident(0) == list(range(8))
    # the test chunk: queries along u (plus noise), its own keys with a third, longer spike in
    # keys 64-127 of the chunk's tile
    q = spiky(("rescale-q", D), L, H, D, [], [], plus=14.0, dtype=dt)
    k = spiky(("rescale-kc", D), L, H, D, [T + 30], [36.0], dtype=dt)
    v = llsynth.seeded_normal(("rescale-vc", D), (L, H, D), dtype=dt, device="cuda")
    for p in range(2):
        st.attend(0, q, k, v, commit=(p == 1), what="%s: reference max moves (pass %d)" % (kernel, p))
    st.check_state()
    st.check_raw(0)
    # a recache prefill whose later blocks hold the spikes (block-causal, 2-frame blocks)
    R = len(st.orc.recache_frames(0))
    qw = spiky(("rescale-qw", D), R * T, H, D, [], [], plus=14.0, dtype=dt)
    kw = spiky(("rescale-kw", D), R * T, H, D, [2 * T + 3, 5 * T + 100], [10.0, 24.0], dtype=dt)
    vw = llsynth.seeded_normal(("rescale-vw", D), (R * T, H, D), dtype=dt, device="cuda")
    st.recache_attend(0, qw, kw, vw, what="%s: prefill with spikes" % kernel)
    st.check_state()
    st.close()
