"""Python binding of libll, the sm_103a short-window + frame-sink attention library.

Thin ctypes marshalling over the C ABI in ``include/ll.h``: every function here
has the name of the C entry point it calls, checks the tensors it is given
(device, dtype, shape, contiguity), passes raw device pointers and the current
CUDA stream, and turns a non-OK status into :class:`LLError`.  All compute runs
in the library's CUDA kernels; there is no fallback.  PyTorch only supplies
device memory and streams.

The operation ("LongLive: Real-time Interactive Long Video Generation", §3.3
Efficient Long Inference and §3.1 KV Recache): a per-layer KV cache holding S
sink frames that are never evicted plus a rolling window of the W most recent
frames; a chunk of C frames attends to [sink || window || its own K/V] and,
when it commits, enters the window with FIFO eviction; a prompt switch
recomputes the resident frames' K/V in place.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libll.so")

LL_BF16, LL_FP32, LL_BF16_K8, LL_FP8 = 0, 1, 2, 3
STATUS = ["LL_OK", "LL_ERR_INVALID_ARG", "LL_ERR_UNSUPPORTED", "LL_ERR_OOM", "LL_ERR_STATE",
          "LL_ERR_CUDA", "LL_ERR_DEVICE_TIMEOUT"]
(LL_OK, LL_ERR_INVALID_ARG, LL_ERR_UNSUPPORTED, LL_ERR_OOM, LL_ERR_STATE, LL_ERR_CUDA,
 LL_ERR_DEVICE_TIMEOUT) = range(7)

# every symbol include/ll.h declares
EXPORTS = ("ll_status_str", "ll_cache_create", "ll_cache_destroy", "ll_attend_chunk", "ll_recache",
           "ll_recache_attend", "ll_reset", "ll_cache_state", "ll_cache_read", "ll_sync",
           "ll_cache_info", "ll_frame_slot", "ll_resident_frames", "ll_launch_count",
           "ll_debug_inject_stall", "ll_debug_use_simt", "ll_profile_enable", "ll_profile_read",
           "ll_set_output_dtype", "ll_debug_attend_schedule", "ll_attend_chunk_noalloc",
           "ll_set_chunk_mask", "ll_set_recache_scope", "ll_recache_tokens", "ll_debug_pair_kernel",
           "ll_debug_poison", "ll_debug_inject_fault")
LL_KERNEL_ATTEND, LL_KERNEL_PREFILL, LL_KERNEL_COPY = 0, 1, 2
LL_MASK_CHUNK, LL_MASK_FRAME = 0, 1
LL_RECACHE_RESIDENT, LL_RECACHE_WINDOW = 0, 1
LL_FAULT_ALLOC, LL_FAULT_LAUNCH = 1, 2


class LLError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, STATUS[status] if 0 <= status < len(STATUS) else status))


_lib_handle = None


def _lib() -> ctypes.CDLL:
    """Load libll.so (built in-tree); fail loudly when it is missing."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libll.so is not built: run `python -m windowed_sink_attention_ll_b300.build_lib`"
                               " (or __graft_entry__.build())")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        sig = {
            "ll_status_str": (ctypes.c_char_p, [i32]),
            "ll_cache_create": (i32, [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32, i32, i32]),
            "ll_cache_destroy": (None, [vp]),
            "ll_attend_chunk": (i32, [vp, i32, vp, vp, vp, vp, i32, vp]),
            "ll_recache": (i32, [vp, i32, vp, vp, vp]),
            "ll_recache_attend": (i32, [vp, i32, vp, vp, vp, vp, vp]),
            "ll_reset": (i32, [vp]),
            "ll_cache_state": (i32, [vp, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]),
            "ll_cache_read": (i32, [vp, i32, vp, vp]),
            "ll_sync": (i32, [vp]),
            "ll_cache_info": (i32, [vp, ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_size_t),
                                    ctypes.POINTER(i32)]),
            "ll_frame_slot": (i32, [i32, i32, i64]),
            "ll_resident_frames": (i32, [i32, i32, i64, ctypes.POINTER(i64)]),
            "ll_launch_count": (ctypes.c_uint64, []),
            "ll_debug_inject_stall": (i32, [vp, i32, i32]),
            "ll_debug_use_simt": (i32, [vp, i32]),
            "ll_debug_pair_kernel": (i32, [vp, i32]),
            "ll_debug_poison": (i32, [vp, i32]),
            "ll_debug_inject_fault": (i32, [i32, i32]),
            "ll_profile_enable": (i32, [vp, i32]),
            "ll_set_output_dtype": (i32, [vp, i32]),
            "ll_debug_attend_schedule": (i32, [i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32),
                                               ctypes.POINTER(i32), i32, ctypes.POINTER(i32), i32,
                                               ctypes.POINTER(i32)]),
            "ll_profile_read": (i32, [vp, i32, ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double)]),
            "ll_attend_chunk_noalloc": (i32, [vp, vp, vp, i32, i64, vp, vp, i32, vp, i32, i32, vp, vp]),
            "ll_set_chunk_mask": (i32, [vp, i32]),
            "ll_set_recache_scope": (i32, [vp, i32]),
            "ll_recache_tokens": (i32, [vp, i32, ctypes.POINTER(i64)]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib_handle = lib
    return _lib_handle


def _check(status: int, where: str) -> None:
    if status != LL_OK:
        raise LLError(status, where)


class LLCache:
    """Handle of one ll_cache plus its shape (for argument checks)."""

    def __init__(self, ptr, layers, heads, head_dim, tokens_per_frame, sink_frames, window_frames,
                 chunk_frames, dtype):
        self.ptr = ptr
        self.layers, self.heads, self.head_dim = layers, heads, head_dim
        self.T, self.S, self.W, self.C = tokens_per_frame, sink_frames, window_frames, chunk_frames
        self.dtype = dtype
        self.torch_dtype = torch.float32 if dtype == LL_FP32 else torch.bfloat16  # token tensors
        # raw K and V caches (e4m3 caches: their bytes)
        self.k_cache_dtype = torch.uint8 if dtype in (LL_BF16_K8, LL_FP8) else self.torch_dtype
        self.v_cache_dtype = torch.uint8 if dtype == LL_FP8 else self.torch_dtype
        self.out_dtype = self.torch_dtype
        self.device = torch.cuda.current_device() if torch.cuda.is_available() else None

    @property
    def slots(self) -> int:
        return self.S + self.W

    def close(self) -> None:
        if self.ptr:
            _lib().ll_cache_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # convenience methods (same calls as the module functions)
    def attend_chunk(self, layer, q, k, v, out, commit, stream=None):
        return ll_attend_chunk(self, layer, q, k, v, out, commit, stream)

    def recache(self, layer, k_win, v_win, stream=None):
        return ll_recache(self, layer, k_win, v_win, stream)

    def recache_attend(self, layer, q_win, k_win, v_win, out_win, stream=None):
        return ll_recache_attend(self, layer, q_win, k_win, v_win, out_win, stream)

    def reset(self):
        return ll_reset(self)

    def state(self, layer):
        return ll_cache_state(self, layer)

    def read(self, layer):
        return ll_cache_read(self, layer)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(cache: LLCache, t, tokens: int, name: str) -> int:
    """Device pointer of a [tokens, H, d] tensor in the cache dtype (outputs: the output dtype)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if cache.device is not None and t.device.index != cache.device:
        raise ValueError("%s is on cuda:%s; the cache lives on cuda:%d" % (name, t.device.index, cache.device))
    want = cache.out_dtype if name.startswith("out") else cache.torch_dtype
    if t.dtype != want:
        raise ValueError("%s has dtype %s, expected %s" % (name, t.dtype, want))
    if tuple(t.shape) != (tokens, cache.heads, cache.head_dim):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape),
                                                          (tokens, cache.heads, cache.head_dim)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def ll_status_str(status: int) -> str:
    return _lib().ll_status_str(status).decode()


def ll_cache_create(layers, heads, head_dim, tokens_per_frame, sink_frames, window_frames, chunk_frames,
                    dtype=LL_BF16) -> LLCache:
    if isinstance(dtype, torch.dtype):
        dtype = LL_BF16 if dtype == torch.bfloat16 else LL_FP32 if dtype == torch.float32 else -1
    out = ctypes.c_void_p()
    _check(_lib().ll_cache_create(ctypes.byref(out), layers, heads, head_dim, tokens_per_frame, sink_frames,
                                  window_frames, chunk_frames, dtype), "ll_cache_create")
    return LLCache(out.value, layers, heads, head_dim, tokens_per_frame, sink_frames, window_frames,
                   chunk_frames, dtype)


def ll_cache_destroy(cache: LLCache) -> None:
    cache.close()


def ll_attend_chunk(cache: LLCache, layer: int, q, k, v, out, commit: bool, stream=None) -> None:
    L = cache.C * cache.T
    args = [_ptr(cache, t, L, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"))]
    _check(_lib().ll_attend_chunk(cache.ptr, layer, *args, 1 if commit else 0, _stream(stream)),
           "ll_attend_chunk")


def ll_recache_tokens(cache: LLCache, layer: int) -> int:
    """Token rows a recache of `layer` reads now (R * T; 0 when the recache would be refused)."""
    n = ctypes.c_int64()
    _check(_lib().ll_recache_tokens(cache.ptr, layer, ctypes.byref(n)), "ll_recache_tokens")
    return n.value


def _recache_rows(cache: LLCache, layer: int, t, name: str) -> int:
    """Rows of a recache window tensor, checked against what the library will read."""
    L = t.shape[0] if isinstance(t, torch.Tensor) and t.dim() > 0 else -1
    want = ll_recache_tokens(cache, layer)
    if want and L != want:
        raise ValueError("%s has %d token rows; a recache of layer %d reads %d" % (name, L, layer, want))
    return L


def ll_recache(cache: LLCache, layer: int, k_win, v_win, stream=None) -> None:
    L = _recache_rows(cache, layer, k_win, "k_win")
    _check(_lib().ll_recache(cache.ptr, layer, _ptr(cache, k_win, L, "k_win"), _ptr(cache, v_win, L, "v_win"),
                             _stream(stream)), "ll_recache")


def ll_recache_attend(cache: LLCache, layer: int, q_win, k_win, v_win, out_win, stream=None) -> None:
    L = _recache_rows(cache, layer, q_win, "q_win")
    ptrs = [_ptr(cache, t, L, n) for t, n in ((q_win, "q_win"), (k_win, "k_win"), (v_win, "v_win"),
                                              (out_win, "out_win"))]
    _check(_lib().ll_recache_attend(cache.ptr, layer, *ptrs, _stream(stream)), "ll_recache_attend")


def ll_reset(cache: LLCache) -> None:
    _check(_lib().ll_reset(cache.ptr), "ll_reset")


def ll_cache_state(cache: LLCache, layer: int):
    """(frames committed, frame_of_slot list); synchronises the device."""
    n = ctypes.c_int64()
    table = (ctypes.c_int64 * max(1, cache.slots))()
    _check(_lib().ll_cache_state(cache.ptr, layer, ctypes.byref(n), table), "ll_cache_state")
    return n.value, [table[i] for i in range(cache.slots)]


def ll_cache_read(cache: LLCache, layer: int):
    """Raw K and V of one layer as CPU tensors [H, S+W, T, d] (synchronises); an
    LL_BF16_K8 cache's K (an LL_FP8 cache's K and V) comes back as e4m3 bytes (torch.uint8)."""
    shape = (cache.heads, cache.slots, cache.T, cache.head_dim)
    hk = torch.empty(shape, dtype=cache.k_cache_dtype)
    hv = torch.empty(shape, dtype=cache.v_cache_dtype)
    _check(_lib().ll_cache_read(cache.ptr, layer, hk.data_ptr(), hv.data_ptr()), "ll_cache_read")
    return hk, hv


def ll_sync(cache: LLCache) -> None:
    _check(_lib().ll_sync(cache.ptr), "ll_sync")


def ll_cache_info(cache: LLCache):
    slots, eb = ctypes.c_int(), ctypes.c_int()
    nbytes = ctypes.c_size_t()
    _check(_lib().ll_cache_info(cache.ptr, ctypes.byref(slots), ctypes.byref(nbytes), ctypes.byref(eb)),
           "ll_cache_info")
    return slots.value, nbytes.value, eb.value


def ll_frame_slot(sink_frames: int, window_frames: int, f: int) -> int:
    return _lib().ll_frame_slot(sink_frames, window_frames, f)


def ll_resident_frames(sink_frames: int, window_frames: int, n: int) -> list:
    buf = (ctypes.c_int64 * max(1, sink_frames + window_frames))()
    cnt = _lib().ll_resident_frames(sink_frames, window_frames, n, buf)
    return [buf[i] for i in range(cnt)]


def ll_resident_count(sink_frames: int, window_frames: int, n: int) -> int:
    return len(ll_resident_frames(sink_frames, window_frames, n))


def ll_launch_count() -> int:
    return _lib().ll_launch_count()


def ll_debug_inject_stall(cache: LLCache, enable: bool, timeout_us: int) -> None:
    _check(_lib().ll_debug_inject_stall(cache.ptr, 1 if enable else 0, timeout_us), "ll_debug_inject_stall")


def ll_debug_use_simt(cache: LLCache, enable: bool) -> None:
    _check(_lib().ll_debug_use_simt(cache.ptr, 1 if enable else 0), "ll_debug_use_simt")


def ll_debug_pair_kernel(cache: LLCache, enable: bool) -> None:
    """head_dim 128 on the CTA-pair tensor-core kernel instead of the one-CTA kernel (test hook)."""
    _check(_lib().ll_debug_pair_kernel(cache.ptr, 1 if enable else 0), "ll_debug_pair_kernel")


def ll_debug_poison(cache: LLCache, enable: bool) -> None:
    """Fill the slots that hold no resident frame with NaN bytes, now and after every reset (test hook)."""
    _check(_lib().ll_debug_poison(cache.ptr, 1 if enable else 0), "ll_debug_poison")


def ll_debug_inject_fault(kind: int, n: int) -> None:
    """Make the n-th next allocation (LL_FAULT_ALLOC) or launch step (LL_FAULT_LAUNCH) fail (0: disarm)."""
    _check(_lib().ll_debug_inject_fault(kind, n), "ll_debug_inject_fault")


def ll_profile_enable(cache: LLCache, enable, every: int = 1) -> None:
    """Time one launch in every `every` of each kind (enable=False: off)."""
    _check(_lib().ll_profile_enable(cache.ptr, max(1, int(every)) if enable else 0), "ll_profile_enable")


def ll_profile_read(cache: LLCache, kind: int):
    """(launches, summed device milliseconds) of one kernel kind; synchronises."""
    n = ctypes.c_int64()
    ms = ctypes.c_double()
    _check(_lib().ll_profile_read(cache.ptr, kind, ctypes.byref(n), ctypes.byref(ms)), "ll_profile_read")
    return n.value, ms.value


def ll_set_output_dtype(cache: LLCache, dtype) -> None:
    """Element type of later outputs: LL_FP32 / torch.float32, or the cache dtype."""
    if isinstance(dtype, torch.dtype):
        dtype = LL_BF16 if dtype == torch.bfloat16 else LL_FP32 if dtype == torch.float32 else -1
    _check(_lib().ll_set_output_dtype(cache.ptr, dtype), "ll_set_output_dtype")
    cache.out_dtype = torch.float32 if dtype == LL_FP32 else torch.bfloat16


def ll_set_chunk_mask(cache: LLCache, mode) -> None:
    """LL_MASK_CHUNK / "chunk" (default) or LL_MASK_FRAME / "frame" (see include/ll.h)."""
    mode = {"chunk": LL_MASK_CHUNK, "frame": LL_MASK_FRAME}.get(mode, mode)
    _check(_lib().ll_set_chunk_mask(cache.ptr, mode), "ll_set_chunk_mask")
    cache.chunk_mask = mode


def ll_set_recache_scope(cache: LLCache, scope) -> None:
    """LL_RECACHE_RESIDENT / "resident" (default) or LL_RECACHE_WINDOW / "window" (see include/ll.h)."""
    scope = {"resident": LL_RECACHE_RESIDENT, "window": LL_RECACHE_WINDOW}.get(scope, scope)
    _check(_lib().ll_set_recache_scope(cache.ptr, scope), "ll_set_recache_scope")
    cache.recache_scope = scope


def ll_debug_attend_schedule(Lq: int, La: int, Lb: int, heads: int, max_ctas: int, mode: int = 0,
                             block_tokens: int = 1):
    """Host replay of a tensor-core attend (mode 0), prefill (mode 1) or frame-causal chunk (mode 2)
    launch's schedule (see include/ll.h).

    Returns (grid, pieces, splits): pieces = list of (cta, item, j0, j1, partial,
    slot); splits = list of (item, [slots of its parts]).
    """
    cap, scap = 6 * 65536, 65536
    pieces = (ctypes.c_int * cap)()
    splits = (ctypes.c_int * scap)()
    grid, nints = ctypes.c_int(), ctypes.c_int()
    n = _lib().ll_debug_attend_schedule(Lq, La, Lb, heads, max_ctas, mode, block_tokens, ctypes.byref(grid), pieces,
                                        cap, splits, scap, ctypes.byref(nints))
    if n < 0:
        raise LLError(LL_ERR_INVALID_ARG, "ll_debug_attend_schedule")
    out = [tuple(pieces[6 * i:6 * i + 6]) for i in range(n)]
    sp, i = [], 0
    while i < nints.value:
        cnt = splits[i + 1]
        sp.append((splits[i], list(splits[i + 2:i + 2 + cnt])))
        i += 2 + cnt
    return grid.value, out, sp


def ll_attend_chunk_noalloc(q, k_cached, v_cached, cached_tokens: int, k, v, out, err_word=None,
                            stream=None) -> None:
    """Chunk attention without any device allocation (see include/ll.h).

    q, k, v, out: contiguous bf16 CUDA tensors [chunk_tokens, H, d].
    k_cached, v_cached: bf16 CUDA tensors [H, rows, d] with contiguous rows per
    head (rows >= cached_tokens), e.g. a layer of ll_cache_read reshaped to
    [H, (S+W)*T, d]; None when cached_tokens is 0.  err_word: optional int32
    CUDA tensor of one element that a timed-out device wait sets to 1.
    """
    L, H, d = (tuple(q.shape) + (0, 0, 0))[:3]
    # the library runs on the current device and encodes every pointer into that device's
    # tensor maps, so every tensor must live there
    dev = torch.cuda.current_device()

    def on_dev(t):
        return t.device.index == dev

    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
                and tuple(t.shape) == (L, H, d) and on_dev(t)):
            raise ValueError("%s must be a contiguous bf16 tensor of shape %s on cuda:%d" % (n, (L, H, d), dev))
    kc = vc = None
    stride = 0
    if cached_tokens > 0:
        for t, n in ((k_cached, "k_cached"), (v_cached, "v_cached")):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.dim() == 3
                    and t.shape[0] == H and t.shape[1] >= cached_tokens and t.shape[2] == d
                    and t.stride(2) == 1 and t.stride(1) == d and on_dev(t)):
                raise ValueError("%s must be a bf16 tensor [H, >= cached_tokens, d] with contiguous rows on cuda:%d"
                                 % (n, dev))
        if k_cached.stride(0) != v_cached.stride(0):
            raise ValueError("k_cached and v_cached must have the same head stride")
        kc, vc, stride = k_cached.data_ptr(), v_cached.data_ptr(), k_cached.stride(0)
    ew = None
    if err_word is not None:
        if not (isinstance(err_word, torch.Tensor) and err_word.is_cuda and err_word.dtype == torch.int32
                and err_word.numel() >= 1 and on_dev(err_word)):
            raise ValueError("err_word must be an int32 tensor of at least one element on cuda:%d" % dev)
        ew = err_word.data_ptr()
    _check(_lib().ll_attend_chunk_noalloc(q.data_ptr(), kc, vc, cached_tokens, stride, k.data_ptr(), v.data_ptr(),
                                          L, out.data_ptr(), H, d, ew, _stream(stream)),
           "ll_attend_chunk_noalloc")
