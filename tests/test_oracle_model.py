"""Pins of the oracle's model math (M1-M3) against things other than itself.

* an fp64 numpy re-evaluation of the whole decoder, written as whole-sequence
  matrix algebra with a causal mask (a different formulation from the oracle's
  per-row loops), itself checked against torch's scaled_dot_product_attention;
* textbook properties of RoPE (identity at position 0, norm preservation,
  scores that depend only on the relative offset);
* RMSNorm's closed form on a constant vector.
"""
import numpy as np
import pytest

import la_inputs as I
import oracle as O

SMALL = I.ModelConfig("small-gqa", 2, 64, 4, 2, 16, 96, 50)


def rope64(x, pos, theta, hd):
    """fp64 rotate-half rotary embedding of x[..., hd] at positions pos[...]."""
    half = hd // 2
    inv = theta ** (-2.0 * np.arange(half) / hd)
    ang = np.asarray(pos, np.float64)[:, None] * inv[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    c = c[:, None, :]
    s = s[:, None, :]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def forward64(cfg, w, tokens):
    """fp64 causal forward of a token sequence at positions 0..n-1 -> logits [n][V]."""
    n = len(tokens)
    H, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    f = lambda a: np.asarray(a, np.float64)
    x = f(w["emb"])[tokens]
    pos = np.arange(n)
    mask = np.tril(np.ones((n, n), bool))

    def norm(v, g):
        return v / np.sqrt((v * v).mean(-1, keepdims=True) + cfg.rms_eps) * f(g)

    for l in range(cfg.n_layers):
        h = norm(x, w["attn_norm"][l])
        q = (h @ f(w["wq"][l]).T).reshape(n, H, hd)
        k = (h @ f(w["wk"][l]).T).reshape(n, Hkv, hd)
        v = (h @ f(w["wv"][l]).T).reshape(n, Hkv, hd)
        q, k = rope64(q, pos, cfg.rope_theta, hd), rope64(k, pos, cfg.rope_theta, hd)
        rep = H // Hkv
        k, v = np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1)
        s = np.einsum("qhd,khd->hqk", q, k) / np.sqrt(hd)
        s = np.where(mask[None], s, -np.inf)
        p = np.exp(s - s.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        o = np.einsum("hqk,khd->qhd", p, v).reshape(n, H * hd)
        x = x + o @ f(w["wo"][l]).T
        h = norm(x, w["ffn_norm"][l])
        g, u = h @ f(w["wg"][l]).T, h @ f(w["wu"][l]).T
        x = x + (g / (1.0 + np.exp(-g)) * u) @ f(w["wd"][l]).T
    return norm(x, w["final_norm"]) @ f(w["lm_head"]).T


def test_reference_attention_matches_torch_sdpa():
    """The fp64 reference's attention equals torch's library routine."""
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(0)
    n, H, hd = 9, 3, 16
    q, k, v = (g.standard_normal((n, H, hd)) for _ in range(3))
    s = np.einsum("qhd,khd->hqk", q, k) / np.sqrt(hd)
    s = np.where(np.tril(np.ones((n, n), bool))[None], s, -np.inf)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    ours = np.einsum("hqk,khd->qhd", p, v)
    t = lambda a: torch.from_numpy(a.transpose(1, 0, 2).copy())
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True)
    np.testing.assert_allclose(ours, ref.numpy().transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("cfg,bf16", [(I.MODELS["tiny"], False), (I.MODELS["tiny"], True), (SMALL, False)])
def test_greedy_logits_match_fp64(cfg, bf16):
    w = I.make_weights(cfg, 0, bf16=bf16)
    m = O.Model(cfg, w)
    prompt = I.random_prompt(12, cfg.vocab, 5)
    toks, lg = O.greedy(m, prompt, 10, logits=True)
    seq = np.concatenate([prompt, toks[:-1]])
    ref = forward64(cfg, w, seq)[len(prompt) - 1:]
    err = np.linalg.norm(lg - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert err.max() < 1e-5, err.max()
    # the emitted tokens are the argmax of those logits
    assert (np.argmax(ref, axis=1) == toks).all()


def test_rope_textbook_properties():
    cfg = SMALL
    m = O.Model(cfg, I.make_weights(cfg, 0))
    s = O.Seq(m, 256)
    c, sn = s.rope_table()
    assert (c[0] == 1.0).all() and (sn[0] == 0.0).all()
    g = np.random.default_rng(1)
    q, k = g.standard_normal(cfg.head_dim).astype(np.float32), g.standard_normal(cfg.head_dim).astype(np.float32)
    assert np.array_equal(s.rope(q, 0), q)
    for p in (1, 17, 200):
        np.testing.assert_allclose(np.linalg.norm(s.rope(q, p)), np.linalg.norm(q), rtol=1e-5)
    # relative-position property: <R(m)q, R(n)k> depends only on m - n
    base = float(np.dot(s.rope(q, 10), s.rope(k, 3)))
    for shift in (1, 50, 180):
        np.testing.assert_allclose(float(np.dot(s.rope(q, 10 + shift), s.rope(k, 3 + shift))), base,
                                   rtol=1e-4, atol=1e-4)
    # and it is not trivially constant
    assert abs(float(np.dot(s.rope(q, 10), s.rope(k, 9))) - base) > 1e-3


def test_first_token_attention_is_its_own_value():
    """With one visible key, attention returns that key's value exactly:
    the oracle's first-position logits equal the fp64 forward of a one-token
    sequence (softmax of a single score is 1)."""
    cfg = SMALL
    w = I.make_weights(cfg, 0)
    m = O.Model(cfg, w)
    s = O.Seq(m, 8)
    lg, _ = s.step(0, [7], [0], [[1]])
    ref = forward64(cfg, w, np.array([7]))
    np.testing.assert_allclose(lg, ref, rtol=1e-5, atol=1e-6)


def test_oracle_attention_matches_fp64_masked_softmax():
    """om_attention against a dense fp64 formulation: keys = cache [0,P) then
    the step rows, with an explicit mask matrix and a library softmax."""
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(4)
    T, H, Hkv, hd, P, max_seq = 9, 4, 2, 16, 11, 32
    q = g.standard_normal((T, H, hd)).astype(np.float32)
    kc = g.standard_normal((Hkv, max_seq, hd)).astype(np.float32)
    vc = g.standard_normal((Hkv, max_seq, hd)).astype(np.float32)
    ks = g.standard_normal((T, Hkv, hd)).astype(np.float32)
    vs = g.standard_normal((T, Hkv, hd)).astype(np.float32)
    k = O.Controller(2, 3, 2, 16)
    k.init(np.arange(16, dtype=np.int32), seed=0)
    for i in range(2):
        k.insert(1, [i + 2, i + 5])
    tok, pos, vis = k.rows(1, P)
    assert len(tok) == T
    out = O.attention(q, kc, vc, ks, vs, vis, pos, P)
    ref = np.zeros_like(out, dtype=np.float64)
    for h in range(H):
        kvh = h // (H // Hkv)
        keys = np.concatenate([kc[kvh, :P], ks[:, kvh]]).astype(np.float64)
        vals = np.concatenate([vc[kvh, :P], vs[:, kvh]]).astype(np.float64)
        mask = np.concatenate([np.ones((T, P), bool), vis.astype(bool)], axis=1)
        s = torch.from_numpy(q[:, h].astype(np.float64) @ keys.T / np.sqrt(hd))
        s = s.masked_fill(~torch.from_numpy(mask), float("-inf"))
        ref[:, h] = torch.softmax(s, dim=-1).numpy() @ vals
    np.testing.assert_allclose(out, ref, rtol=1e-5, atol=1e-5)
