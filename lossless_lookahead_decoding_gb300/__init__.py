"""Python binding of liblookahead.so (include/lookahead.h).

Argument marshalling only: every step of the decode path runs in the library's
CUDA kernels.  PyTorch is used for device memory (weights, workspace) and
streams.  The functions keep the C names (``la_create``, ``la_prefill``,
``la_step``, ``la_generate``, ...); ``Decoder`` bundles a model description,
its device weights and a context.

Importing this package does not need a GPU; calling into the library does.  If
the shared library has not been built, every call raises -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblookahead.so")

LA_OK, LA_ERR_ARG, LA_ERR_OOM, LA_ERR_CAPACITY, LA_ERR_CUDA, LA_ERR_TIMEOUT, LA_ERR_STATE = 0, -1, -2, -3, -4, -5, -6
LA_FP32, LA_BF16 = 0, 1
LA_PRESEED_PROMPT, LA_DEBUG_LOGITS, LA_NO_GRAPH, LA_SIMT, LA_PROFILE, LA_ATTN_TC, LA_MASK_DIAG = 1, 2, 4, 8, 16, 32, 64

EXPORTS = ("la_workspace_bytes", "la_create", "la_prefill", "la_step", "la_generate", "la_set_sampling", "la_get_stats",
           "la_get_profile", "la_set_top_k", "la_set_top_p", "la_workspace_bytes_batch", "la_create_batch", "la_prefill_seq", "la_step_batch",
           "la_generate_batch",
           "la_debug_logits", "la_debug_argmax", "la_debug_rows", "la_debug_pool", "la_debug_window",
           "la_debug_set_argmax_override", "la_debug_select",
           "la_last_error", "la_destroy", "la_attention", "la_attention_noalloc", "la_pool_create", "la_pool_insert", "la_pool_lookup", "la_pool_size",
           "la_pool_destroy")


class LAError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{msg} (code {code})")
        self.code = code


class la_model_desc(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("d_model", C.c_int), ("n_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn", C.c_int), ("vocab", C.c_int), ("max_seq", C.c_int),
                ("rms_eps", C.c_float), ("rope_theta", C.c_float), ("dtype", C.c_int),
                ("emb", C.c_void_p), ("layer_w", C.c_void_p), ("final_norm", C.c_void_p),
                ("lm_head", C.c_void_p), ("stream", C.c_void_p)]


class la_stats(C.Structure):
    _fields_ = [("steps", C.c_longlong), ("emitted", C.c_longlong), ("prefill_tokens", C.c_longlong),
                ("accept_hist", C.c_longlong * 9), ("P", C.c_int), ("rows", C.c_int),
                ("last_step_ms", C.c_float), ("kernels_per_step", C.c_int)]


class la_prof_entry(C.Structure):
    _fields_ = [("name", C.c_char * 24), ("launches", C.c_longlong), ("total_ms", C.c_double),
                ("bytes", C.c_double), ("flops", C.c_double)]


_lib = None


def lib():
    """Load liblookahead.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run lossless_lookahead_decoding_gb300/build.py "
                               "(there is no fallback implementation)")
        L = C.CDLL(LIB_PATH)
        vp, i32, sz, u64 = C.c_void_p, C.c_int, C.c_size_t, C.c_uint64
        sig = {
            "la_workspace_bytes": (sz, [vp, i32, i32, i32]),
            "la_create": (i32, [vp, i32, i32, i32, vp, sz, u64, i32, vp]),
            "la_prefill": (i32, [vp, vp, i32]),
            "la_step": (i32, [vp, vp, i32, vp]),
            "la_generate": (i32, [vp, vp, i32, i32, vp, vp]),
            "la_workspace_bytes_batch": (sz, [vp, i32, i32, i32, i32]),
            "la_create_batch": (i32, [vp, i32, i32, i32, i32, vp, sz, u64, i32, vp]),
            "la_prefill_seq": (i32, [vp, i32, vp, i32]),
            "la_step_batch": (i32, [vp, vp, i32, vp]),
            "la_generate_batch": (i32, [vp, vp, vp, i32, vp, vp]),
            "la_debug_select": (i32, [vp, i32]),
            "la_set_sampling": (i32, [vp, C.c_float, u64]),
            "la_set_top_k": (i32, [vp, i32]), "la_set_top_p": (i32, [vp, C.c_float]),
            "la_get_stats": (i32, [vp, vp]),
            "la_get_profile": (i32, [vp, vp, i32, vp]),
            "la_debug_logits": (i32, [vp, vp, sz]),
            "la_debug_argmax": (i32, [vp, vp, i32, vp]),
            "la_debug_rows": (i32, [vp, vp, vp, i32, vp, vp]),
            "la_debug_pool": (i32, [vp, i32, vp, i32, vp]),
            "la_debug_window": (i32, [vp, vp, i32]),
            "la_debug_set_argmax_override": (i32, [vp, vp, i32]),
            "la_last_error": (C.c_char_p, [vp]),
            "la_destroy": (None, [vp]),
            "la_attention": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp]),
            "la_attention_noalloc": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp]),
            "la_pool_create": (i32, [i32, i32, i32, vp, vp]),
            "la_pool_insert": (i32, [vp, vp, vp, i32]),
            "la_pool_lookup": (i32, [vp, vp, i32, vp, vp]),
            "la_pool_size": (i32, [vp, vp]),
            "la_pool_destroy": (None, [vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _check(ctx, rc):
    if rc != LA_OK:
        msg = lib().la_last_error(ctx).decode() if ctx else "error"
        raise LAError(rc, msg)


# ------------------------------------------------------------- C entry points

def la_workspace_bytes(desc: la_model_desc, W: int, N: int, G: int) -> int:
    return int(lib().la_workspace_bytes(C.byref(desc), W, N, G))


def la_create(desc: la_model_desc, W: int, N: int, G: int, workspace: int = 0, ws_bytes: int = 0,
              seed: int = 2, flags: int = 0):
    h = C.c_void_p()
    rc = lib().la_create(C.byref(desc), W, N, G, workspace or None, ws_bytes, seed, flags, C.byref(h))
    if rc != LA_OK:
        raise LAError(rc, "la_create failed")
    return h


def la_prefill(ctx, prompt) -> None:
    p = np.ascontiguousarray(prompt, dtype=np.int32)
    _check(ctx, lib().la_prefill(ctx, _p(p), len(p)))


def la_step(ctx, N: int = 8) -> np.ndarray:
    out = np.zeros(max(N, 8), np.int32)
    n = C.c_int()
    _check(ctx, lib().la_step(ctx, _p(out), len(out), C.byref(n)))
    return out[: n.value].copy()


def la_workspace_bytes_batch(desc: la_model_desc, W: int, N: int, G: int, batch: int) -> int:
    return int(lib().la_workspace_bytes_batch(C.byref(desc), W, N, G, batch))


def la_create_batch(desc: la_model_desc, W: int, N: int, G: int, batch: int, workspace: int = 0, ws_bytes: int = 0,
                    seed: int = 2, flags: int = 0):
    h = C.c_void_p()
    rc = lib().la_create_batch(C.byref(desc), W, N, G, batch, workspace or None, ws_bytes, seed, flags, C.byref(h))
    if rc != LA_OK:
        raise LAError(rc, "la_create_batch failed")
    return h


def la_prefill_seq(ctx, seq: int, prompt) -> None:
    p = np.ascontiguousarray(prompt, dtype=np.int32)
    _check(ctx, lib().la_prefill_seq(ctx, seq, _p(p), len(p)))


def la_step_batch(ctx, batch: int, N: int = 8) -> list:
    """One step of every sequence: a list of `batch` token arrays."""
    cap = max(N, 8)
    out = np.zeros((batch, cap), np.int32)
    n = np.zeros(batch, np.int32)
    _check(ctx, lib().la_step_batch(ctx, _p(out), cap, _p(n)))
    return [out[b, : n[b]].copy() for b in range(batch)]


def la_generate_batch(ctx, prompts, max_new: int) -> list:
    """Prefill every sequence with its prompt and step until each has max_new
    tokens: a list of token arrays, one per sequence."""
    ps = [np.ascontiguousarray(p, dtype=np.int32) for p in prompts]
    flat = np.ascontiguousarray(np.concatenate(ps), dtype=np.int32)
    lens = np.array([len(p) for p in ps], np.int32)
    out = np.zeros((len(ps), max(max_new, 1)), np.int32)
    n = np.zeros(len(ps), np.int32)
    _check(ctx, lib().la_generate_batch(ctx, _p(flat), _p(lens), max_new, _p(out), _p(n)))
    return [out[b, : n[b]].copy() for b in range(len(ps))]


def la_debug_select(ctx, seq: int) -> None:
    _check(ctx, lib().la_debug_select(ctx, seq))


def la_set_sampling(ctx, temperature: float, seed: int) -> None:
    _check(ctx, lib().la_set_sampling(ctx, float(temperature), int(seed)))


def la_set_top_k(ctx, top_k: int) -> None:
    _check(ctx, lib().la_set_top_k(ctx, int(top_k)))


def la_set_top_p(ctx, top_p: float) -> None:
    _check(ctx, lib().la_set_top_p(ctx, float(top_p)))


def la_generate(ctx, prompt, max_new: int) -> np.ndarray:
    p = np.ascontiguousarray(prompt, dtype=np.int32)
    out = np.zeros(max(max_new, 1), np.int32)
    n = C.c_int()
    _check(ctx, lib().la_generate(ctx, _p(p), len(p), max_new, _p(out), C.byref(n)))
    return out[: n.value].copy()


def la_get_stats(ctx) -> dict:
    s = la_stats()
    _check(ctx, lib().la_get_stats(ctx, C.byref(s)))
    return {"steps": s.steps, "emitted": s.emitted, "prefill_tokens": s.prefill_tokens,
            "accept_hist": list(s.accept_hist), "P": s.P, "rows": s.rows, "last_step_ms": s.last_step_ms,
            "kernels_per_step": s.kernels_per_step}


def la_get_profile(ctx) -> dict:
    arr = (la_prof_entry * 16)()
    n = C.c_int()
    _check(ctx, lib().la_get_profile(ctx, arr, 16, C.byref(n)))
    return {arr[i].name.decode(): {"launches": arr[i].launches, "total_ms": arr[i].total_ms,
                                   "bytes": arr[i].bytes, "flops": arr[i].flops} for i in range(n.value)}


def la_debug_logits(ctx, T: int, V: int) -> np.ndarray:
    out = np.zeros((T, V), np.float32)
    _check(ctx, lib().la_debug_logits(ctx, _p(out), out.size))
    return out


def la_debug_argmax(ctx, cap: int = 128) -> np.ndarray:
    out = np.zeros(cap, np.int32)
    T = C.c_int()
    _check(ctx, lib().la_debug_argmax(ctx, _p(out), cap, C.byref(T)))
    return out[: T.value].copy()


def la_debug_rows(ctx, cap: int = 128):
    tok = np.zeros(cap, np.int32)
    pos = np.zeros(cap, np.int32)
    T, nc = C.c_int(), C.c_int()
    _check(ctx, lib().la_debug_rows(ctx, _p(tok), _p(pos), cap, C.byref(T), C.byref(nc)))
    return tok[: T.value].copy(), pos[: T.value].copy(), nc.value


def la_debug_pool(ctx, key: int, G: int, N: int) -> np.ndarray:
    out = np.zeros(max(G, 1) * (N - 1), np.int32)
    n = C.c_int()
    _check(ctx, lib().la_debug_pool(ctx, key, _p(out), len(out), C.byref(n)))
    return out[: n.value * (N - 1)].reshape(n.value, N - 1).copy()


def la_debug_window(ctx, W: int, N: int) -> np.ndarray:
    out = np.zeros(max(W * (N - 1), 1), np.int32)
    _check(ctx, lib().la_debug_window(ctx, _p(out), len(out)))
    return out[: W * (N - 1)].reshape(N - 1, W).copy()


def la_debug_set_argmax_override(ctx, amax) -> None:
    """amax: one token per step row, or None to clear the override."""
    if amax is None:
        _check(ctx, lib().la_debug_set_argmax_override(ctx, None, 0))
        return
    a = np.ascontiguousarray(amax, dtype=np.int32)
    _check(ctx, lib().la_debug_set_argmax_override(ctx, _p(a), len(a)))


def la_last_error(ctx) -> str:
    return lib().la_last_error(ctx).decode()


def la_destroy(ctx) -> None:
    if ctx:
        lib().la_destroy(ctx)


def la_attention(q, k_cache, v_cache, k_step, v_step, out, n_heads, n_kv_heads, head_dim, max_seq, P, W, N, G,
                 stream: int = 0) -> int:
    """Pointers are device addresses (ints); returns the C status code."""
    return lib().la_attention(q, k_cache, v_cache, k_step, v_step, out, n_heads, n_kv_heads, head_dim, max_seq, P,
                              W, N, G, stream or None)


def la_attention_noalloc(q, k_cache, v_cache, k_step, v_step, out, n_heads, n_kv_heads, head_dim, max_seq, P, W,
                         N, G, stream: int = 0) -> int:
    """la_attention with its scratch in the library's fixed device array (no
    device allocation); returns the C status code."""
    return lib().la_attention_noalloc(q, k_cache, v_cache, k_step, v_step, out, n_heads, n_kv_heads, head_dim,
                                      max_seq, P, W, N, G, stream or None)


def la_pool_create(capacity: int, N: int, G: int, stream: int = 0):
    h = C.c_void_p()
    rc = lib().la_pool_create(capacity, N, G, stream or None, C.byref(h))
    if rc != LA_OK:
        raise LAError(rc, "la_pool_create failed")
    return h


def la_pool_insert(pool, keys_ptr: int, grams_ptr: int, n: int) -> int:
    return lib().la_pool_insert(pool, keys_ptr, grams_ptr, n)


def la_pool_lookup(pool, keys_ptr: int, n: int, out_ptr: int, counts_ptr: int) -> int:
    return lib().la_pool_lookup(pool, keys_ptr, n, out_ptr, counts_ptr)


def la_pool_size(pool) -> int:
    n = C.c_int()
    rc = lib().la_pool_size(pool, C.byref(n))
    if rc:
        raise LAError(rc, "la_pool_size failed")
    return n.value


def la_pool_destroy(pool) -> None:
    if pool:
        lib().la_pool_destroy(pool)


# ------------------------------------------------------------------ Decoder

LAYER_ORDER = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")


def device_weights(cfg, tensors, dtype: int, device="cuda"):
    """Upload fp32 host arrays (``name -> array`` or ``name -> [per layer]``,
    the la_inputs layout) to device tensors of the model dtype.  Accepts an
    iterator of (name, layer, array) to stream large models."""
    import torch
    tdt = torch.bfloat16 if dtype == LA_BF16 else torch.float32
    out = {n: [None] * cfg.n_layers for n in LAYER_ORDER}
    items = tensors if not isinstance(tensors, dict) else (
        [(n, -1, tensors[n]) for n in ("emb", "final_norm", "lm_head")] +
        [(n, l, tensors[n][l]) for n in LAYER_ORDER for l in range(cfg.n_layers)])
    for name, layer, a in items:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device).to(tdt)
        if layer >= 0:
            out[name][layer] = t
        else:
            out[name] = t
    return out


class Decoder:
    """A model description + device weights + one decoding context (batch > 1:
    a batched context of that many sequences, see ``la_create_batch``)."""

    def __init__(self, cfg, weights, dtype: int, W: int, N: int, G: int, max_seq: int, seed: int = 2,
                 flags: int = 0, stream=None, batch: int = 1):
        import torch
        self.cfg, self.W, self.N, self.G, self.dtype, self.flags = cfg, W, N, G, dtype, flags
        self.w = weights
        self._ptrs = (C.c_void_p * (cfg.n_layers * 9))(
            *[weights[n][l].data_ptr() for l in range(cfg.n_layers) for n in LAYER_ORDER])
        # a non-default stream: the step is captured into a CUDA graph, which
        # the legacy default stream does not allow
        self.stream = stream if stream is not None else torch.cuda.Stream()
        torch.cuda.synchronize()
        self.desc = la_model_desc(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn,
                                  cfg.vocab, max_seq, cfg.rms_eps, cfg.rope_theta, dtype,
                                  weights["emb"].data_ptr(), C.cast(self._ptrs, C.c_void_p).value,
                                  weights["final_norm"].data_ptr(), weights["lm_head"].data_ptr(),
                                  self.stream.cuda_stream)
        self.T = 1 + (W + G) * (N - 1)
        self.batch = batch
        self.ctx = (la_create(self.desc, W, N, G, 0, 0, seed, flags) if batch == 1 else
                    la_create_batch(self.desc, W, N, G, batch, 0, 0, seed, flags))

    def close(self):
        if getattr(self, "ctx", None):
            la_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        self.close()

    def prefill(self, prompt):
        la_prefill(self.ctx, prompt)

    def step(self):
        return la_step(self.ctx, self.N)

    def prefill_seq(self, seq: int, prompt):
        la_prefill_seq(self.ctx, seq, prompt)

    def step_batch(self):
        return la_step_batch(self.ctx, self.batch, self.N)

    def generate_batch(self, prompts, max_new: int):
        return la_generate_batch(self.ctx, prompts, max_new)

    def select(self, seq: int):
        """Point the debug accessors at sequence seq."""
        la_debug_select(self.ctx, seq)

    def set_sampling(self, temperature: float, seed: int, top_k: int = 0, top_p: float = 1.0):
        """Sampling verification at this temperature (<= 0: greedy), from each
        row's top_k tokens when top_k > 0, then from the leading ones holding
        top_p of their weight when top_p < 1."""
        la_set_sampling(self.ctx, temperature, seed)
        la_set_top_k(self.ctx, top_k)
        la_set_top_p(self.ctx, top_p)

    def generate(self, prompt, max_new: int):
        return la_generate(self.ctx, prompt, max_new)

    def stats(self):
        return la_get_stats(self.ctx)

    def profile(self):
        return la_get_profile(self.ctx)

    def logits(self):
        return la_debug_logits(self.ctx, self.T, self.cfg.vocab)

    def argmax(self):
        return la_debug_argmax(self.ctx)

    def rows(self):
        return la_debug_rows(self.ctx)

    def pool(self, key: int):
        return la_debug_pool(self.ctx, key, self.G, self.N)

    def window(self):
        return la_debug_window(self.ctx, self.W, self.N)

    def override_argmax(self, amax):
        la_debug_set_argmax_override(self.ctx, amax)
