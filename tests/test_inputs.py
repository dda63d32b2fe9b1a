"""The seeded input generators (la_inputs): the recipe both the oracle and the
GPU path read their weights and prompts from.

* bf16 rounding equals torch's round-to-nearest-even cast (so host-rounded
  weights and weights cast on the device hold the same bytes);
* Zipf tokens follow P(k) proportional to (k+1)^-s;
* planted spans are exact copies of earlier windows, at least the requested
  number of them;
* weights are deterministic, N(0, 0.02^2) with unit norm weights, and a layer
  slice holds the same bytes as the full model's layers;
* each workload's prompt has the stated length and id range.
"""
import numpy as np
import pytest
import torch

import la_inputs as I


def test_bf16_round_matches_torch_cast():
    g = np.random.default_rng(0)
    x = np.concatenate([
        g.standard_normal(100_000).astype(np.float32) * np.float32(3.0),
        g.standard_normal(1000).astype(np.float32) * np.float32(1e-38),   # subnormals
        g.standard_normal(1000).astype(np.float32) * np.float32(1e37),
        # exact halfway cases, both parities of the kept bit
        (np.arange(1, 2001, dtype=np.uint32) << np.uint32(16) | np.uint32(0x8000)).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0], np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = I.bf16_round(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(I.bf16_bits(got).astype(np.uint32) << np.uint32(16), got.view(np.uint32))


def test_zipf_tokens_follow_the_power_law():
    n, vocab, s = 200_000, 1000, 1.1
    t = I.zipf_tokens(n, vocab, s, 3)
    assert t.dtype == np.int32 and t.min() >= 0 and t.max() < vocab
    k = np.arange(1, vocab + 1, dtype=np.float64)
    p = k ** -s / (k ** -s).sum()
    freq = np.bincount(t, minlength=vocab) / n
    for i in range(5):
        assert abs(freq[i] - p[i]) <= 5 * np.sqrt(p[i] * (1 - p[i]) / n), (i, freq[i], p[i])
    assert np.array_equal(t, I.zipf_tokens(n, vocab, s, 3))


@pytest.mark.parametrize("workload,n,vocab,copies", [("tiny", 32, 1024, 2), ("7b", 512, 32000, 6),
                                                    ("13b", 1024, 32000, 13), ("34b", 2048, 4000, 51)])
def test_prompts_and_planted_spans(workload, n, vocab, copies):
    p = I.make_prompt(workload)
    assert p.dtype == np.int32 and len(p) == n and p.min() >= 0 and p.max() < vocab
    assert np.array_equal(p, I.make_prompt(workload))
    span = 8 if workload == "tiny" else 16
    copied = 0
    for b in range(1, n // span):
        blk = p[b * span:(b + 1) * span]
        if any(np.array_equal(blk, p[s:s + span]) for s in range(0, b * span - span + 1)):
            copied += 1
    assert copied >= copies


def test_weights_recipe_and_slices():
    cfg = I.MODELS["tiny"]
    w = I.make_weights(cfg, 0)
    w2 = I.make_weights(cfg, 0)
    for name in ("emb", "lm_head", "final_norm"):
        assert np.array_equal(w[name], w2[name])
    for name in I.LAYER_TENSORS:
        for l in range(cfg.n_layers):
            assert np.array_equal(w[name][l], w2[name][l])
            if name.endswith("norm"):
                assert (w[name][l] == 1).all()
    big = w["lm_head"]
    assert abs(float(big.std()) - 0.02) < 1e-3 and abs(float(big.mean())) < 1e-3
    # a slice of the model holds the same bytes as the full model's layers
    sl = I.make_weights(cfg, 0, layers=[1])
    for name in I.LAYER_TENSORS:
        assert np.array_equal(sl[name][1], w[name][1]) and sl[name][0] is None
    # bf16 weights are the rounding of the fp32 draws
    wb = I.make_weights(cfg, 0, bf16=True)
    assert np.array_equal(wb["wq"][0], I.bf16_round(w["wq"][0]))
