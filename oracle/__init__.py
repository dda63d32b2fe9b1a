"""CPU oracle for Lookahead Decoding -- TEST INFRASTRUCTURE.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may
import this package.  It wraps ``oracle.c`` (plain fp32 C, no BLAS, built with
``-O2 -fno-fast-math -ffp-contract=off``; OpenMP only over independent output
elements, so results do not depend on the thread count) through ctypes.  It
shares no code with the CUDA library.

Functions and what pins them (the tests under tests/test_oracle_*.py):
  greedy          plain greedy decoding -- pinned by an fp64 numpy/torch
                  re-evaluation of the layer math, textbook special cases of
                  RMSNorm/RoPE/softmax, and the library routine
                  ``scaled_dot_product_attention``.
  lookahead       the method -- pinned by losslessness (equal to greedy token
                  for token, the summary's exactness claim), the step shape
                  T = 1 + (W+G)(N-1) against the pages' 120x/80x/56x FLOPs
                  figures, per-row equivalence of the masked forward with the
                  plain causal forward, a brute-force LCP check of verification
                  and a list-based replay of the pool.
  Controller      the window/pool/verify state machine fed external argmaxes
                  (or, for sampling verification, the rows' logits).
  sample_decode / lookahead_sample / sample_logits
                  temperature sampling and the sampling verification (R10) --
                  pinned by an exact rational enumeration of the verification
                  rule, Monte-Carlo agreement of the oracle's draws with the
                  softmax and, on a Markov toy model, of the sampled lookahead's
                  token sequences with plain ancestral sampling's exact
                  probabilities, and the tau -> 0 reduction to greedy decoding.
  The "diagonal levels" mask reading R3' (variant=DIAGONAL) is pinned the
  same way: losslessness, a brute-force walk of its visibility sets with the
  gap-free invariant, per-row equivalence with the causal forward and a
  list-based replay of its diagonal harvest and Jacobi window update.
  Parity unpinned: acceptance rate and the choice among the readings R1, R3,
  R3', R6, R7 (nothing on the pages fixes them).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP)."""
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
                               "-fPIC", "-shared", "-fvisibility=hidden", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Model(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("d_model", C.c_int), ("n_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("ffn", C.c_int),
                ("vocab", C.c_int), ("rms_eps", C.c_float), ("rope_theta", C.c_float),
                ("emb", C.c_void_p), ("final_norm", C.c_void_p), ("lm_head", C.c_void_p),
                ("attn_norm", C.c_void_p), ("wq", C.c_void_p), ("wk", C.c_void_p),
                ("wv", C.c_void_p), ("wo", C.c_void_p), ("ffn_norm", C.c_void_p),
                ("wg", C.c_void_p), ("wu", C.c_void_p), ("wd", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        vp, i32, u64, f32, f64 = C.c_void_p, C.c_int, C.c_uint64, C.c_float, C.c_double
        sig = {
            "om_seq_new": (vp, [vp, i32]), "om_seq_free": (None, [vp]),
            "om_threads": (i32, []), "om_set_threads": (None, [i32]), "om_rope_table": (None, [vp, vp, vp]),
            "om_rope": (None, [vp, vp, i32]),
            "om_step_forward": (i32, [vp, i32, i32, vp, vp, vp, vp, vp]),
            "om_commit": (i32, [vp, i32, i32, vp]), "om_prefill": (i32, [vp, i32, vp, i32]),
            "om_greedy": (i32, [vp, vp, i32, i32, i32, vp, vp]),
            "om_ctrl_new": (vp, [i32, i32, i32, i32]), "om_ctrl_free": (None, [vp]),
            "om_splitmix64": (u64, [vp]), "om_pool_insert": (None, [vp, i32, vp]),
            "om_ctrl_init": (i32, [vp, vp, i32, u64, i32]), "om_ctrl_rows_max": (i32, [vp]),
            "om_ctrl_rows": (i32, [vp, i32, i32, vp, vp, vp]),
            "om_ctrl_advance": (i32, [vp, vp, vp, vp, vp]), "om_ctrl_pool": (i32, [vp, i32, vp]),
            "om_ctrl_window": (None, [vp, vp]),
            "om_lookahead": (i32, [vp, vp, i32, i32, i32, i32, u64, i32, i32, i32, i32, vp, vp, vp]),
            "om_ctrl_set_variant": (i32, [vp, i32]),
            "om_attention": (i32, [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]),
            "om_uniform": (f64, [vp]), "om_exp_neg": (f32, [f32]),
            "om_sample_weight": (C.c_uint64, [f32, f32, f32, i32]),
            "om_sample_logits": (None, [vp, i32, f32, i32, f32, vp, i32, vp]),
            "om_ctrl_advance_sample": (i32, [vp, vp, f32, i32, f32, vp, vp, vp, vp]),
            "om_sample_decode": (i32, [vp, vp, i32, i32, i32, f32, i32, f32, u64, vp]),
            "om_top_k_key": (u64, [u64, i32, i32]), "om_top_p24": (C.c_uint32, [f32]),
            "om_lookahead_sample": (i32, [vp, vp, i32, i32, i32, i32, u64, i32, i32, f32, i32, f32, u64, i32, i32, vp,
                                          vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class Model:
    """fp32 host copy of a decoder's weights, in the oracle's struct."""

    def __init__(self, cfg, weights):
        self.cfg = cfg
        f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
        self._keep = []

        def arr(x):
            x = f32(x)
            self._keep.append(x)
            return x.ctypes.data

        def per_layer(name):
            ptrs = (C.c_void_p * cfg.n_layers)(*[arr(w) for w in weights[name]])
            self._keep.append(ptrs)
            return C.cast(ptrs, C.c_void_p).value

        self.s = _Model(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                        cfg.ffn, cfg.vocab, cfg.rms_eps, cfg.rope_theta,
                        arr(weights["emb"]), arr(weights["final_norm"]), arr(weights["lm_head"]),
                        *[per_layer(n) for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm",
                                                 "wg", "wu", "wd")])

    @property
    def ptr(self):
        return C.cast(C.pointer(self.s), C.c_void_p)


class Seq:
    """A KV cache plus the step forward of the oracle."""

    def __init__(self, model: Model, max_seq: int):
        self.model = model
        self.max_seq = max_seq
        self.h = lib().om_seq_new(model.ptr, max_seq)
        if not self.h:
            raise MemoryError("om_seq_new failed")

    def __del__(self):
        if getattr(self, "h", None):
            lib().om_seq_free(self.h)
            self.h = None

    def prefill(self, toks, P0: int = 0):
        t = _i32(toks)
        if lib().om_prefill(self.h, P0, _p(t), len(t)):
            raise ValueError("om_prefill failed")

    def step(self, P: int, tok, pos, vis, want_logits: bool = True):
        tok, pos = _i32(tok), _i32(pos)
        T = len(tok)
        vis = np.ascontiguousarray(np.asarray(vis, dtype=np.uint8).reshape(T, T))
        logits = np.zeros((T, self.model.cfg.vocab), np.float32) if want_logits else None
        amax = np.zeros(T, np.int32)
        rc = lib().om_step_forward(self.h, P, T, _p(tok), _p(pos), _p(vis),
                                   _p(logits) if want_logits else None, _p(amax))
        if rc:
            raise ValueError("om_step_forward failed")
        return logits, amax

    def commit(self, P: int, rows):
        r = _i32(rows)
        if lib().om_commit(self.h, P, len(r), _p(r)):
            raise ValueError("om_commit failed")

    def rope(self, v, pos: int):
        x = np.ascontiguousarray(np.asarray(v, dtype=np.float32)).copy()
        lib().om_rope(self.h, _p(x), pos)
        return x

    def rope_table(self):
        half = self.model.cfg.head_dim // 2
        c = np.zeros((self.max_seq, half), np.float32)
        s = np.zeros((self.max_seq, half), np.float32)
        lib().om_rope_table(self.h, _p(c), _p(s))
        return c, s


def greedy(model: Model, prompt, max_new: int, max_seq: int | None = None, logits: bool = False):
    p = _i32(prompt)
    max_seq = max_seq or (len(p) + max_new + 8)
    out = np.zeros(max_new, np.int32)
    lg = np.zeros((max_new, model.cfg.vocab), np.float32) if logits else None
    if lib().om_greedy(model.ptr, _p(p), len(p), max_new, max_seq, _p(out), _p(lg) if logits else None):
        raise ValueError("om_greedy failed")
    return (out, lg) if logits else out


DIAGONAL = 1  # mask reading R3' ("diagonal levels"); 0 is R3


def lookahead(model: Model, prompt, W: int, N: int, G: int, max_new: int, seed: int = 2,
              preseed: bool = False, max_seq: int | None = None, variant: int = 0):
    """Returns (tokens, steps, accept_hist[0..N]).  variant: 0 = mask reading
    R3, DIAGONAL = R3'."""
    p = _i32(prompt)
    max_seq = max_seq or (len(p) + max_new + W + N + 8)
    out = np.zeros(max_new, np.int32)
    steps = np.zeros(1, np.int32)
    hist = np.zeros(N + 1, np.int32)
    rc = lib().om_lookahead(model.ptr, _p(p), len(p), W, N, G, seed, int(preseed), variant, max_new, max_seq,
                            _p(out), _p(steps), _p(hist))
    if rc:
        raise ValueError("om_lookahead failed")
    return out, int(steps[0]), hist


def sample_decode(model: Model, prompt, max_new: int, tau: float, rng_seed: int, max_seq: int | None = None,
                  top_k: int = 0, top_p: float = 1.0):
    """Plain ancestral sampling at temperature tau (top_k > 0: from the top_k
    tokens by weight; top_p < 1: then from the smallest leading set of those
    holding top_p of their weight)."""
    p = _i32(prompt)
    max_seq = max_seq or (len(p) + max_new + 8)
    out = np.zeros(max_new, np.int32)
    if lib().om_sample_decode(model.ptr, _p(p), len(p), max_new, max_seq, tau, top_k, top_p, rng_seed, _p(out)):
        raise ValueError("om_sample_decode failed")
    return out


def lookahead_sample(model: Model, prompt, W: int, N: int, G: int, max_new: int, tau: float, rng_seed: int,
                     seed: int = 2, preseed: bool = False, max_seq: int | None = None, variant: int = 0,
                     top_k: int = 0, top_p: float = 1.0):
    """Lookahead decoding with sampling verification; (tokens, steps, accept_hist)."""
    p = _i32(prompt)
    max_seq = max_seq or (len(p) + max_new + W + N + 8)
    out = np.zeros(max_new, np.int32)
    steps = np.zeros(1, np.int32)
    hist = np.zeros(N + 1, np.int32)
    rc = lib().om_lookahead_sample(model.ptr, _p(p), len(p), W, N, G, seed, int(preseed), variant, tau, top_k,
                                   top_p, rng_seed, max_new, max_seq, _p(out), _p(steps), _p(hist))
    if rc:
        raise ValueError("om_lookahead_sample failed")
    return out, int(steps[0]), hist


class Rng:
    """The splitmix64 stream the sampling functions draw their uniforms from."""

    def __init__(self, seed: int):
        self.state = (C.c_uint64 * 1)(seed)

    @property
    def ptr(self):
        return C.cast(self.state, C.c_void_p)

    def uniform(self) -> float:
        return lib().om_uniform(self.ptr)


def exp_neg(x: float) -> float:
    """The fp32 exponential (x <= 0) of the sampling probabilities."""
    return lib().om_exp_neg(float(x))


def sample_weight(z: float, mx: float, tau: float, V: int) -> int:
    """Integer weight floor(exp((z - mx) / tau) 2^B) of a token, B = 63 -
    ceil(log2(V + 1)): p(v) = weight / sum of weights."""
    return int(lib().om_sample_weight(float(z), float(mx), float(tau), int(V)))


def sample_logits(z, tau: float, rng: Rng, n: int, top_k: int = 0, top_p: float = 1.0):
    """n draws from softmax(z / tau) (one uniform each); top_k > 0: from the
    top_k tokens by weight, ties to the lower index; top_p < 1: then from the
    smallest leading set of those, in the same order, holding at least top_p
    of their weight."""
    z = np.ascontiguousarray(z, dtype=np.float32)
    out = np.zeros(n, np.int32)
    lib().om_sample_logits(_p(z), len(z), tau, top_k, top_p, rng.ptr, n, _p(out))
    return out


def top_p24(top_p: float) -> int:
    """The top-p bound as floor(top_p 2^24) in 1..2^24 (2^24: no restriction)."""
    return int(lib().om_top_p24(float(top_p)))


def top_k_key(E: int, v: int, V: int) -> int:
    """The order of the top-k restriction: E(v) V + (V - 1 - v)."""
    return int(lib().om_top_k_key(int(E), int(v), int(V)))


def splitmix64_stream(seed: int, n: int):
    st = (C.c_uint64 * 1)(seed)
    return [lib().om_splitmix64(C.cast(st, C.c_void_p)) for _ in range(n)]


class Controller:
    """Window / pool / verification state machine (R1-R9) fed external argmaxes."""

    def __init__(self, W: int, N: int, G: int, V: int, variant: int = 0):
        self.W, self.N, self.G, self.V, self.variant = W, N, G, V, variant
        self.h = lib().om_ctrl_new(W, N, G, V)
        if not self.h or lib().om_ctrl_set_variant(self.h, variant):
            raise ValueError("bad controller arguments")
        self.Tmax = lib().om_ctrl_rows_max(self.h)

    def __del__(self):
        if getattr(self, "h", None):
            lib().om_ctrl_free(self.h)
            self.h = None

    def init(self, prompt, seed: int = 2, preseed: bool = False):
        p = _i32(prompt)
        lib().om_ctrl_init(self.h, _p(p), len(p), seed, int(preseed))

    def insert(self, key: int, val):
        v = _i32(val)
        lib().om_pool_insert(self.h, key, _p(v))

    def rows(self, c: int, P: int):
        tok = np.zeros(self.Tmax, np.int32)
        pos = np.zeros(self.Tmax, np.int32)
        vis = np.zeros(self.Tmax * self.Tmax, np.uint8)
        T = lib().om_ctrl_rows(self.h, c, P, _p(tok), _p(pos), _p(vis))
        return tok[:T].copy(), pos[:T].copy(), vis[:T * T].reshape(T, T).copy()

    def advance(self, amax):
        a = _i32(amax)
        emit = np.zeros(self.N + 1, np.int32)
        rows = np.zeros(self.N + 1, np.int32)
        g = (C.c_int * 1)()
        n = lib().om_ctrl_advance(self.h, _p(a), _p(emit), _p(rows), C.cast(g, C.c_void_p))
        return emit[:n].copy(), rows[:n].copy(), int(g[0])

    def advance_sample(self, logits, tau: float, rng: Rng, top_k: int = 0, top_p: float = 1.0):
        """R10 verification by sampling from the rows' logits [T][V] (top_k >
        0: each row restricted to its top_k tokens; top_p < 1: then to the
        leading set holding top_p of their weight), then the R6/R7 harvest
        and shift with the rows' argmaxes."""
        lg = np.ascontiguousarray(logits, dtype=np.float32)
        emit = np.zeros(self.N + 1, np.int32)
        rows = np.zeros(self.N + 1, np.int32)
        g = (C.c_int * 1)()
        n = lib().om_ctrl_advance_sample(self.h, _p(lg), tau, top_k, top_p, rng.ptr, _p(emit), _p(rows),
                                         C.cast(g, C.c_void_p))
        return emit[:n].copy(), rows[:n].copy(), int(g[0])

    def pool(self, key: int):
        out = np.zeros(max(self.G, 1) * (self.N - 1), np.int32)
        n = lib().om_ctrl_pool(self.h, key, _p(out))
        return out[: n * (self.N - 1)].reshape(n, self.N - 1).copy()

    def window(self):
        out = np.zeros(max(self.W, 1) * (self.N - 1), np.int32)
        lib().om_ctrl_window(self.h, _p(out))
        return out[: self.W * (self.N - 1)].reshape(self.N - 1, self.W).copy()


def attention(q, k_cache, v_cache, k_step, v_step, vis, pos, P: int):
    """One layer's masked attention: q [T][H][hd], k/v_cache [Hkv][max_seq][hd]
    (positions [0,P) used), k/v_step [T][Hkv][hd], vis [T][T], pos [T] ->
    out [T][H][hd] (fp32)."""
    f = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    q, kc, vc, ks, vs = f(q), f(k_cache), f(v_cache), f(k_step), f(v_step)
    T, H, hd = q.shape
    Hkv, max_seq = kc.shape[0], kc.shape[1]
    vis = np.ascontiguousarray(np.asarray(vis, dtype=np.uint8).reshape(T, T))
    pos = _i32(pos)
    out = np.zeros((T, H, hd), np.float32)
    if lib().om_attention(T, H, Hkv, hd, max_seq, P, _p(q), _p(kc), _p(vc), _p(ks), _p(vs), _p(vis), _p(pos),
                          _p(out)):
        raise ValueError("om_attention failed")
    return out


def threads() -> int:
    return lib().om_threads()


def set_threads(n: int) -> None:
    """Threads of the oracle's parallel loops (results do not depend on it)."""
    lib().om_set_threads(int(n))
