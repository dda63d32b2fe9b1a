"""Seeded synthetic inputs shared by the CUDA path's tests/bench and by the CPU oracle.

This module holds no arithmetic of the decoding method: it only draws random
weights, prompts and attention-benchmark tensors from fixed seeds, so that the
oracle and the CUDA library can be fed the very same bytes.

Workload shapes follow the lookahead-decoding summary page (Fu et al. 2024,
"Break the Sequential Dependency of LLM Inference Using Lookahead Decoding",
Key points: 7B W=15 N=5, 13B W=10 N=5, 34B W=7 N=5, G=W) with Llama-style
decoders of those sizes; models are random-init and prompts are synthetic
Zipf draws with planted repeated spans (the pages' chat/code suites are not
reproduced).

Seeds: weights seed 0, prompt seed 1, window seed 2 by default.  Per-tensor
seed = base + index of the tensor in the fixed order
emb, per layer (attn_norm, wq, wk, wv, wo, ffn_norm, wg, wu, wd), final_norm,
lm_head.  Every matrix ~ N(0, 0.02^2), drawn in fp32 and (for bf16 models)
rounded to bf16 round-to-nearest-even; norm weights are 1.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0

    @property
    def d_kv(self) -> int:
        return self.n_kv_heads * self.head_dim

    def shapes(self):
        """(name, layer, shape) in the fixed generation order."""
        d, f, q, kv = self.d_model, self.ffn, self.n_heads * self.head_dim, self.d_kv
        out = [("emb", -1, (self.vocab, d))]
        per = {"attn_norm": (d,), "wq": (q, d), "wk": (kv, d), "wv": (kv, d),
               "wo": (d, q), "ffn_norm": (d,), "wg": (f, d), "wu": (f, d), "wd": (d, f)}
        for layer in range(self.n_layers):
            out += [(n, layer, per[n]) for n in LAYER_TENSORS]
        out += [("final_norm", -1, (d,)), ("lm_head", -1, (self.vocab, d))]
        return out

    def streamed_params(self) -> int:
        """Parameters one decode step streams: every layer matrix + LM head."""
        d, f, q, kv = self.d_model, self.ffn, self.n_heads * self.head_dim, self.d_kv
        per_layer = q * d + 2 * kv * d + d * q + 3 * f * d
        return self.n_layers * per_layer + self.vocab * d

    def sliced(self, n_layers: int) -> "ModelConfig":
        return dataclasses.replace(self, name=f"{self.name}-{n_layers}L", n_layers=n_layers)


MODELS = {
    "tiny": ModelConfig("tiny", 2, 256, 4, 4, 64, 688, 1024),
    "7b": ModelConfig("7b", 32, 4096, 32, 32, 128, 11008, 32000),
    "13b": ModelConfig("13b", 40, 5120, 40, 40, 128, 13824, 32000),
    "34b": ModelConfig("34b", 48, 8192, 64, 8, 128, 22016, 32000),
}

# (W, N, G) per workload, from the pages' near-optimal A100 settings (G = W)
# and the tiny case.
LOOKAHEAD = {"tiny": (4, 3, 4), "7b": (15, 5, 15), "13b": (10, 5, 10), "34b": (7, 5, 7)}


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns fp32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) & np.uint32(0xFFFF0000)).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of already bf16-exact fp32 values."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _draw(shape, seed: int, std: float = 0.02) -> np.ndarray:
    g = np.random.default_rng(seed)
    return g.standard_normal(shape, dtype=np.float32) * np.float32(std)


def iter_weights(cfg: ModelConfig, seed: int = 0, bf16: bool = True, layers=None, threads=None):
    """Yield (name, layer, fp32 array) in the fixed order.

    ``layers`` restricts which decoder layers are drawn (the others are
    skipped; their seeds are still reserved, so a slice of a model holds the
    same bytes as the full model's layers).
    Arrays hold bf16-exact values when ``bf16`` is set.
    """
    items = []
    for idx, (name, layer, shape) in enumerate(cfg.shapes()):
        if layer >= 0 and layers is not None and layer not in layers:
            continue
        items.append((idx, name, layer, shape))

    def make(item):
        idx, name, layer, shape = item
        if name.endswith("norm"):
            a = np.ones(shape, dtype=np.float32)
        else:
            a = _draw(shape, seed + idx)
            if bf16:
                a = bf16_round(a)
        return name, layer, a

    threads = threads or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(threads) as ex:
        # keep at most ``threads`` tensors in flight so big models stream
        pending = []
        for it in items:
            pending.append(ex.submit(make, it))
            if len(pending) >= threads:
                yield pending.pop(0).result()
        for p in pending:
            yield p.result()


def make_weights(cfg: ModelConfig, seed: int = 0, bf16: bool = False, layers=None):
    """All weights as a dict: emb, final_norm, lm_head, and per-layer lists."""
    w = {n: [None] * cfg.n_layers for n in LAYER_TENSORS}
    for name, layer, a in iter_weights(cfg, seed, bf16, layers):
        if layer >= 0:
            w[name][layer] = a
        else:
            w[name] = a
    return w


def zipf_tokens(n: int, vocab: int, s: float, seed: int) -> np.ndarray:
    """n tokens with P(k) proportional to (k+1)^-s, k = 0..vocab-1, id = k."""
    k = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(k ** -s)
    cdf /= cdf[-1]
    u = np.random.default_rng(seed).random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1).astype(np.int32)


def plant_spans(tokens: np.ndarray, span: int, copies: int, seed: int) -> np.ndarray:
    """Copy ``copies`` earlier spans of length ``span`` onto distinct later
    span-aligned destination blocks (each source starts before its block)."""
    t = tokens.copy()
    n_blocks = len(t) // span
    if copies <= 0 or n_blocks < 2:
        return t
    g = np.random.default_rng(seed)
    dests = np.sort(g.choice(np.arange(1, n_blocks), size=min(copies, n_blocks - 1), replace=False))
    for b in dests:
        dst = int(b) * span
        src = int(g.integers(0, dst - span + 1))
        t[dst:dst + span] = t[src:src + span]
    return t


def make_prompt(workload: str, seed: int = 1) -> np.ndarray:
    """The synthetic prompt of a named workload."""
    if workload == "tiny":
        return plant_spans(zipf_tokens(32, 1024, 1.1, seed), 8, 2, seed + 1000)
    if workload == "7b":
        return plant_spans(zipf_tokens(512, 32000, 1.1, seed), 16, round(0.2 * 512 / 16), seed + 1000)
    if workload == "13b":
        return plant_spans(zipf_tokens(1024, 32000, 1.1, seed), 16, round(0.2 * 1024 / 16), seed + 1000)
    if workload == "34b":
        return plant_spans(zipf_tokens(2048, 4000, 1.2, seed), 16, round(0.4 * 2048 / 16), seed + 1000)
    raise KeyError(workload)


def random_prompt(n: int, vocab: int, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).integers(0, vocab, n).astype(np.int32)


def attention_bench_inputs(seed: int = 3, heads: int = 32, head_dim: int = 128, ctx: int = 2048,
                           rows: int = 121):
    """Attention micro-benchmark tensors: K/V cache [heads][ctx][hd] ~ N(0,1),
    step Q/K/V [rows][heads][hd] ~ N(0,1), all bf16-exact fp32."""
    g = np.random.default_rng(seed)
    f = lambda *s: bf16_round(g.standard_normal(s, dtype=np.float32))
    return {"k_cache": f(heads, ctx, head_dim), "v_cache": f(heads, ctx, head_dim),
            "q": f(rows, heads, head_dim), "k_step": f(rows, heads, head_dim),
            "v_step": f(rows, heads, head_dim)}


def pool_bench_ngrams(n: int, vocab: int = 32000, n_minus_1: int = 4, s: float = 1.1, seed: int = 4):
    """n (key, (N-1)-gram) pairs with Zipf(s) tokens for the pool micro-bench."""
    toks = zipf_tokens(n * (1 + n_minus_1), vocab, s, seed).reshape(n, 1 + n_minus_1)
    return toks[:, 0].copy(), toks[:, 1:].copy()


def pool_bench_inserts(n_keys: int = 4096, per_key: int = 20, vocab: int = 32000, n_minus_1: int = 4,
                       s: float = 1.1, seed: int = 5):
    """Insert stream for the pool micro-benchmark: n_keys distinct Zipf(s) keys,
    per_key Zipf(s) (N-1)-grams each, in a seeded interleaved order.
    Returns keys int32[n], grams int32[n][N-1]."""
    g = np.random.default_rng(seed)
    keys, seen, draw = [], set(), 0
    while len(keys) < n_keys:
        for t in zipf_tokens(4 * n_keys, vocab, s, seed + 17 + draw).tolist():
            if t not in seen:
                seen.add(t)
                keys.append(t)
                if len(keys) == n_keys:
                    break
        draw += 1
    k = np.repeat(np.array(keys, np.int32), per_key)
    order = g.permutation(len(k))
    grams = zipf_tokens(len(k) * n_minus_1, vocab, s, seed + 1).reshape(len(k), n_minus_1)
    return k[order].copy(), grams.astype(np.int32)
