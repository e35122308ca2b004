"""Two caches driven from two host threads on two CUDA streams at the same time.

The C ABI allows concurrent calls on different caches (calls on one cache are
not thread-safe): each cache keeps its own host bookkeeping, and the library's
shared state (launch counter, fault countdowns, per-device attribute flags) is
atomic.  Here two threads each stream chunks through their own cache on their
own stream, so their kernels interleave on the device, and every output, the
cache state and the raw slot bytes must match a float64 oracle of that thread's
own calls ("LongLive", §3.3 "Frame sink" + "Short window attention"), within
max |err| <= 1e-2 and relative L2 <= 5e-3.
"""

import threading

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


class StreamLockstep(Lockstep):
    """Lockstep whose library calls go to one CUDA stream."""

    def __init__(self, *args, stream, **kw):
        super().__init__(*args, **kw)
        self.stream = stream

    def attend(self, layer, q, k, v, commit, rows=None, check=True, what=""):
        with torch.cuda.stream(self.stream):
            out = torch.empty(q.shape, dtype=self.cache.out_dtype, device=q.device)
            self.ll.ll_attend_chunk(self.cache, layer, q, k, v, out, commit, self.stream)
        self.stream.synchronize()
        return self._check_after(layer, q, k, v, out, commit, rows, check, what)

    def _check_after(self, layer, q, k, v, out, commit, rows, check, what):
        if check:
            from tests.gpu_util import compare

            want = self.orc.attend(layer, self.qk64(q), self.qk64(k), self.v64(v), commit, rows=rows)
            compare(out, want, what)
        elif commit:
            self.orc.commit(layer, self.qk64(k), self.v64(v))
        if commit and self.keep:
            t0 = self.orc.state(layer)[0] - self.C
            kc, vc = self.key_store(k), self.value_store(v)
            for i in range(self.C):
                self.host[layer][t0 + i] = (kc[i * self.T:(i + 1) * self.T], vc[i * self.T:(i + 1) * self.T])
        return out


def drive(ll, kind, errors):
    try:
        torch.cuda.set_device(0)
        stream = torch.cuda.Stream()
        H, D, T, S, W, C = (6, 128, 200, 3, 6, 3) if kind == "bf16" else (5, 128, 150, 2, 4, 2)
        st = StreamLockstep(ll, 2, H, D, T, S, W, C, torch.bfloat16, value_fp8=(kind == "fp8"), stream=stream)
        L = C * T
        for c in range(6):
            for layer in (0, 1):
                with torch.cuda.stream(stream):
                    q, k, v = (llsynth.seeded_normal(("threads", kind, layer, c, t), (L, H, D), device="cuda")
                               for t in "qkv")
                st.attend(layer, q, k, v, commit=True, what="thread %s L%d c%d" % (kind, layer, c))
            st.check_state()
        st.check_raw(0)
        st.check_raw(1)
        st.close()
    except BaseException as e:  # reported by the main thread
        errors.append((kind, e))


def test_two_threads_two_streams(ll):
    errors = []
    threads = [threading.Thread(target=drive, args=(ll, kind, errors)) for kind in ("bf16", "fp8")]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, errors
