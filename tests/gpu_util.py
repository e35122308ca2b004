"""Helpers of the GPU parity tests: a GPU cache driven in lock-step with the oracle."""

import numpy as np
import torch

import oracle

# Tolerance of the attention outputs against the float64 oracle with bf16
# inputs (same for fp32): max |err| <= 1e-2 and relative L2 <= 5e-3.
ATOL = 1e-2
REL_L2 = 5e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 values just above |x| (8 significant bits): the most that
    rounding a value to x can have moved it."""
    ax = np.maximum(np.abs(x), np.finfo(np.float64).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 8)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 values rounded once to the nearest bf16 value (8 significant bits, ties to
    even; the range of the outputs compared here stays far from bf16 overflow/underflow)."""
    f, e = np.frexp(x)  # x = f * 2^e, 0.5 <= |f| < 1
    return np.ldexp(np.round(f * 256.0) / 256.0, e)


# Every comparison's max |err| and relative L2, per test (written out by tests/conftest.py when
# LL_PARITY_LOG names a file).
OBSERVED = []


def compare(got: torch.Tensor, want: np.ndarray, what: str, atol=ATOL, rel_l2=REL_L2):
    """max|err| <= atol and relative L2 <= rel_l2 against the unrounded float64 oracle.

    atol=None is the form for bf16 outputs of large magnitude.  Rounding the exact result
    to bf16 alone can move it by more than 1e-2 there (half an ulp is |o| * 2^-9), and a
    result computed within 1e-2 that lands on the other side of a rounding midpoint from the
    oracle comes out one whole ulp away from bf16(oracle).  The check is then that each
    output is the bf16 rounding of some value within 1e-2 of the oracle,
    |got - oracle| <= 1e-2 + half an ulp of got, and the relative L2 bound against the
    unrounded oracle."""
    g = f64(got)
    assert g.shape == want.shape, (what, g.shape, want.shape)
    assert np.isfinite(g).all(), what + ": non-finite output"
    diff = np.abs(g - want)
    err = float(diff.max())
    rel = float(np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-30))
    rec = {"what": what, "max_abs_err": err, "rel_l2": rel, "max_abs_out": float(np.abs(want).max()),
           "bf16_out": atol is None}
    OBSERVED.append(rec)
    if atol is None:
        excess = float((diff - bf16_half_ulp(g)).max())
        rec["max_err_beyond_rounding"] = excess
        rec["max_abs_err_vs_bf16_oracle"] = float(np.abs(g - round_bf16(want)).max())
        assert excess <= ATOL and rel <= rel_l2, (
            "%s: max(|err| - half ulp of out) %.3e (<= %g), max|err| %.3e, rel_l2 %.3e (<= %g)" % (
                what, excess, ATOL, err, rel, rel_l2))
        return err, rel
    assert err <= atol and rel <= rel_l2, "%s: max|err| %.3e (<= %g), rel_l2 %.3e (<= %g)" % (
        what, err, atol, rel, rel_l2)
    return err, rel


def sample_rows(L: int, n: int, seed: int = 0) -> np.ndarray:
    """Deterministic query-row sample: both ends, tile edges, the ragged tail, random rest."""
    fixed = {0, 1, 127, 128, 255, 256, 383, 384, L - 1, L - 2, (L // 128) * 128, (L // 256) * 256 - 1}
    fixed = {r for r in fixed if 0 <= r < L}
    rng = np.random.default_rng(seed)
    rest = rng.choice(L, size=min(L, max(0, n - len(fixed))), replace=False)
    return np.array(sorted(fixed | set(int(r) for r in rest)), dtype=np.int64)


def bits(t: torch.Tensor) -> torch.Tensor:
    if t.element_size() == 1:
        return t.view(torch.uint8)
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def round_e4m3(t: torch.Tensor) -> torch.Tensor:
    """bf16 values rounded to FP8 e4m3 as the library rounds keys and queries for the
    e4m3 caches (and values for LL_FP8): nearest value, ties to even, saturating at +-448 (torch's own
    conversion returns NaN past 480, hence the clamp).  Returns a float8_e4m3fn CPU tensor."""
    return torch.clamp(t.detach().cpu().float(), -448.0, 448.0).to(torch.float8_e4m3fn)


class Lockstep:
    """A libll cache and an oracle cache fed the same calls; checks state after each one.

    The cache's empty slots are poisoned (NaN bytes, ll_debug_poison), now and after every
    reset: an attention that read a slot holding no resident frame would return NaN.

    ``host`` keeps, per layer and frame, the exact K/V values the GPU was given
    (CPU tensors), so the raw cache bytes can be compared slot by slot.
    """

    def __init__(self, ll, layers, heads, head_dim, T, S, W, C, dtype, keep_frames=True, key_fp8=False,
                 value_fp8=False):
        """key_fp8: an LL_BF16_K8 cache (bf16 tokens, e4m3 key cache); the oracle is fed q and k
        rounded to e4m3 as the library rounds them, and the raw K slots hold e4m3 bytes.
        value_fp8: an LL_FP8 cache (e4m3 keys and values): v is rounded the same way too."""
        self.ll = ll
        self.key_fp8 = key_fp8 or value_fp8
        self.value_fp8 = value_fp8
        code = ll.LL_FP8 if value_fp8 else ll.LL_BF16_K8 if key_fp8 else dtype
        self.cache = ll.ll_cache_create(layers, heads, head_dim, T, S, W, C, code)
        # slots without a resident frame hold NaN bytes, so a read of one would show in the outputs
        ll.ll_debug_poison(self.cache, True)
        self.orc = oracle.OracleCache(layers, heads, head_dim, T, S, W, C)
        self.shape = (layers, heads, head_dim, T, S, W, C)
        self.dtype = dtype
        self.keep = keep_frames
        self.host = [dict() for _ in range(layers)]
        self._zeros = None
        self.atol = ATOL

    @property
    def T(self):
        return self.shape[3]

    @property
    def C(self):
        return self.shape[6]

    def qk64(self, t):
        """q or k as the oracle sees them: rounded to e4m3 first for an FP8-key cache."""
        return f64(round_e4m3(t)) if self.key_fp8 else f64(t)

    def key_store(self, k):
        """What the K cache stores for keys k (CPU): the e4m3 bytes for an FP8-key cache."""
        return round_e4m3(k).view(torch.uint8) if self.key_fp8 else k.cpu()

    def v64(self, t):
        """v as the oracle sees it: rounded to e4m3 first for an LL_FP8 cache."""
        return f64(round_e4m3(t)) if self.value_fp8 else f64(t)

    def value_store(self, v):
        """What the V cache stores for values v (CPU): the e4m3 bytes for an LL_FP8 cache."""
        return round_e4m3(v).view(torch.uint8) if self.value_fp8 else v.cpu()

    def attend(self, layer, q, k, v, commit, rows=None, check=True, what=""):
        """q, k, v: CUDA tensors.  Returns the GPU output (and checks it unless check=False)."""
        out = torch.empty(q.shape, dtype=self.cache.out_dtype, device=q.device)
        self.ll.ll_attend_chunk(self.cache, layer, q, k, v, out, commit)
        if check:
            qh, kh, vh = self.qk64(q), self.qk64(k), self.v64(v)
            want = self.orc.attend(layer, qh, kh, vh, commit, rows=rows)
            got = out if rows is None else out[torch.as_tensor(rows, device=out.device)]
            compare(got, want, what or "attend", atol=self.atol)
        elif commit:
            kh, vh = self.qk64(k), self.v64(v)
            self.orc.commit(layer, kh, vh)
        if commit and self.keep:
            t0 = self.orc.state(layer)[0] - self.C
            kc, vc = self.key_store(k), self.value_store(v)
            for i in range(self.C):
                self.host[layer][t0 + i] = (kc[i * self.T:(i + 1) * self.T], vc[i * self.T:(i + 1) * self.T])
        return out

    def set_options(self, chunk_mask="chunk", recache_scope="resident"):
        """The two optional readings, on the library cache and on the oracle alike."""
        self.ll.ll_set_chunk_mask(self.cache, chunk_mask)
        self.ll.ll_set_recache_scope(self.cache, recache_scope)
        self.orc.set_chunk_mask(chunk_mask)
        self.orc.set_recache_scope(recache_scope)

    def commit_placeholder(self, layer, q, k, v):
        """GPU gets the real chunk; the oracle a zero chunk.

        For chunks whose frames no checked output can see: if the GPU kept such a
        frame by mistake, the checked outputs would differ from the oracle's.
        """
        out = torch.empty(q.shape, dtype=self.cache.out_dtype, device=q.device)
        self.ll.ll_attend_chunk(self.cache, layer, q, k, v, out, True)
        if self._zeros is None or self._zeros.shape != tuple(q.shape):
            self._zeros = np.zeros(tuple(q.shape))
        self.orc.commit(layer, self._zeros, self._zeros)
        return out

    def recache(self, layer, k_win, v_win):
        self.ll.ll_recache(self.cache, layer, k_win, v_win)
        self.orc.recache(layer, self.qk64(k_win), self.v64(v_win))
        self._keep_recache(layer, k_win, v_win)

    def recache_attend(self, layer, q_win, k_win, v_win, rows=None, check=True, what=""):
        out = torch.empty(q_win.shape, dtype=self.cache.out_dtype, device=q_win.device)
        self.ll.ll_recache_attend(self.cache, layer, q_win, k_win, v_win, out)
        if check:
            want = self.orc.recache_attend(layer, self.qk64(q_win), self.qk64(k_win), self.v64(v_win), rows=rows)
            got = out if rows is None else out[torch.as_tensor(rows, device=out.device)]
            compare(got, want, what or "recache prefill", atol=self.atol)
        else:
            self.orc.recache(layer, self.qk64(k_win), self.v64(v_win))
        self._keep_recache(layer, k_win, v_win)
        return out

    def _keep_recache(self, layer, k_win, v_win):
        if not self.keep:
            return
        kc, vc = self.key_store(k_win), self.value_store(v_win)
        for i, f in enumerate(self.orc.recache_frames(layer)):
            self.host[layer][f] = (kc[i * self.T:(i + 1) * self.T], vc[i * self.T:(i + 1) * self.T])

    def check_state(self, layers=None):
        for layer in range(self.shape[0]) if layers is None else layers:
            got = self.ll.ll_cache_state(self.cache, layer)
            assert got == self.orc.state(layer), (layer, got, self.orc.state(layer))

    def check_raw(self, layer):
        """Every occupied slot holds, bit for bit, the K/V the oracle says it holds."""
        hk, hv = self.ll.ll_cache_read(self.cache, layer)
        for slot, f in self.orc.expected_slots(layer).items():
            k, v = self.host[layer][f]
            assert torch.equal(bits(hk[:, slot]), bits(k.permute(1, 0, 2).contiguous())), (layer, slot, f)
            assert torch.equal(bits(hv[:, slot]), bits(v.permute(1, 0, 2).contiguous())), (layer, slot, f)

    def close(self):
        self.cache.close()
