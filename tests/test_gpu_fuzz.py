"""Random call sequences through the C ABI, in lockstep with the oracle.

Each case draws a shape (ragged tokens per frame, any sink / window / chunk
sizes including zero sink and zero window), a dtype (bf16: the tensor-core
kernel; fp32: the tensor-core kernel with tf32 operands at head_dim 64, the
CUDA-core kernel at 128; a second set of cases uses the e4m3 caches, keys or
keys and values, at head_dim 128) and a sequence of calls: committing and
non-committing chunk passes, recache with and without the prefill attention,
reset, and switches of the two optional readings (chunk mask, recache scope)
between calls.  After every call the outputs are compared with the float64
oracle (max |err| <= 1e-2 and relative L2 <= 5e-3, as in the other parity
tests) and the frames committed and the frame-to-slot map must match exactly;
after every call that writes the cache the raw slot bytes of that layer must
match the K/V the oracle says each slot holds, bit for bit.
"""

import numpy as np
import pytest
import torch

import llsynth
from tests.gpu_util import Lockstep

pytestmark = pytest.mark.gpu

CASES = 40
E4M3_CASES = 16
OPS = ["commit", "commit", "commit", "commit", "pass", "pass", "prefill", "recache", "reset", "options"]


@pytest.fixture(scope="module")
def ll():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    torch.cuda.set_device(0)
    return mod


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    shape = dict(
        layers=int(rng.integers(1, 3)),
        H=int(rng.integers(1, 4)),
        D=int(rng.choice([64, 128])),
        T=int(rng.integers(1, 151)),
        S=int(rng.integers(0, 4)),
        W=int(rng.integers(0, 8)),
        C=int(rng.integers(1, 5)),
    )
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    ops = [str(rng.choice(OPS)) for _ in range(int(rng.integers(14, 26)))]
    return rng, shape, dtype, ops


@pytest.mark.parametrize("seed", range(CASES))
def test_random_call_sequence(ll, seed):
    rng, s, dtype, ops = draw_case(seed)
    run_case(ll, seed, rng, s, dtype, ops, None)


@pytest.mark.parametrize("seed", range(CASES, CASES + E4M3_CASES))
def test_random_call_sequence_e4m3_caches(ll, seed):
    """The same kind of sequences on the e4m3 caches (head_dim 128): even seeds store keys in
    e4m3, odd seeds keys and values."""
    rng, s, _, ops = draw_case(seed)
    s["D"] = 128
    run_case(ll, seed, rng, s, torch.bfloat16, ops, "keys" if seed % 2 == 0 else "kv")


def run_case(ll, seed, rng, s, dtype, ops, e4m3):
    H, D, T, S, W, C = s["H"], s["D"], s["T"], s["S"], s["W"], s["C"]
    st = Lockstep(ll, s["layers"], H, D, T, S, W, C, dtype, key_fp8=(e4m3 == "keys"), value_fp8=(e4m3 == "kv"))
    mask, scope = "chunk", "resident"
    L = C * T

    def inputs(tag, rows, names="qkv"):
        return [llsynth.seeded_normal(("fuzz", seed, tag, t), (rows, H, D), dtype=dtype, device="cuda")
                for t in names]

    for i, op in enumerate(ops):
        layer = int(rng.integers(0, s["layers"]))
        what = "seed %d op %d %s layer %d %s %s/%s %s" % (seed, i, op, layer, s, mask, scope, e4m3 or dtype)
        if op in ("commit", "pass"):
            q, k, v = inputs(i, L)
            st.attend(layer, q, k, v, commit=(op == "commit"), what=what)
            if op == "commit":
                st.check_raw(layer)
        elif op in ("prefill", "recache"):
            R = len(st.orc.recache_frames(layer))
            assert ll.ll_recache_tokens(st.cache, layer) == R * T, what
            if R == 0:
                z = torch.zeros((T, H, D), dtype=dtype, device="cuda")
                with pytest.raises(ll.LLError) as e:
                    ll.ll_recache(st.cache, layer, z, z)
                assert e.value.status == ll.LL_ERR_STATE, what
                continue
            if op == "prefill":
                qw, kw, vw = inputs(i, R * T)
                st.recache_attend(layer, qw, kw, vw, what=what)
            else:
                kw, vw = inputs(i, R * T, "kv")
                st.recache(layer, kw, vw)
            st.check_raw(layer)
        elif op == "reset":
            ll.ll_reset(st.cache)
            st.orc.reset()
        else:
            mask = str(rng.choice(["chunk", "frame"]))
            scope = str(rng.choice(["resident", "window"]))
            st.set_options(mask, scope)
        st.check_state()
    st.close()
