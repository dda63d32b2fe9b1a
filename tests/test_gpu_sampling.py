"""GPU sampling verification (la_set_sampling) against the oracle's rule.

The GPU runs the tiny workload with sampling verification; after every step
the oracle controller is fed the GPU's own logits and its uniform stream
(same splitmix64 seed).  The emitted tokens, window and pool must then be
bit-exact: both sides turn the same logits into the same integer weights
(the same fp32 exponential, operation for operation) and take every
accept/reject decision and every draw in exact integer arithmetic.  Also
with the diagonal-levels mask and with the tensor-core attention option.
tau -> 0 must reproduce greedy decoding, and a temperature of 0 must restore
it.
"""
import math

import numpy as np
import pytest

import la_inputs as I
import oracle as O
from helpers import build_lib, gpu_decoder

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()


def _setup(dtype):
    cfg = I.MODELS["tiny"]
    w = I.make_weights(cfg, 0, bf16=dtype == 1)
    return cfg, w, I.make_prompt("tiny"), I.LOOKAHEAD["tiny"]


@pytest.mark.parametrize("dtype,flags,top_k,tau,top_p",
                         [(0, 0, 0, 0.05, 1.0), (1, 0, 0, 0.05, 1.0), (1, 64, 0, 0.05, 1.0), (1, 32, 0, 0.05, 1.0),
                          (0, 0, 5, 0.8, 1.0), (1, 0, 40, 1.0, 1.0), (1, 32, 2, 0.7, 1.0), (1, 0, 1, 1.0, 1.0),
                          (1, 0, 1024, 0.05, 1.0), (0, 0, 0, 0.8, 0.9), (1, 0, 40, 1.0, 0.5), (1, 32, 0, 0.7, 0.95),
                          (1, 64, 0, 2.0, 0.3), (1, 0, 0, 1.0, 1e-6), (1, 0, 3, 1.0, 0.999)],
                         ids=["fp32", "bf16", "bf16-diagonal", "bf16-attntc", "fp32-top5", "bf16-top40",
                              "bf16-attntc-top2", "bf16-top1", "bf16-topV", "fp32-p0.9", "bf16-top40-p0.5",
                              "bf16-attntc-p0.95", "bf16-diagonal-p0.3", "bf16-p-tiny", "bf16-top3-p0.999"])
def test_sampled_steps_replay_the_oracle_rule(dtype, flags, top_k, tau, top_p):
    """(top_k > 0: each row restricted to its top_k tokens by weight, on both
    sides; top_k = vocab keeps every token; top_p < 1: then to the leading
    tokens holding top_p of their weight.)"""
    import lossless_lookahead_decoding_gb300 as LA
    cfg, w, prompt, (W, N, G) = _setup(dtype)
    seed = 77
    dec = gpu_decoder(cfg, w, dtype, W, N, G, 256, flags=flags | LA.LA_DEBUG_LOGITS)
    dec.set_sampling(tau, seed, top_k=top_k, top_p=top_p)
    ctrl = O.Controller(W, N, G, cfg.vocab, variant=O.DIAGONAL if flags & LA.LA_MASK_DIAG else 0)
    ctrl.init(prompt, seed=2)
    rng = O.Rng(seed)
    dec.prefill(prompt)
    assert np.array_equal(dec.window(), ctrl.window())
    c, P, multi = int(prompt[-1]), len(prompt) - 1, 0
    for _ in range(40):
        emit = dec.step()
        tok_g, pos_g, ncand = dec.rows()
        tok, pos, _ = ctrl.rows(c, P)
        T = len(tok)
        assert np.array_equal(tok_g[:T], tok) and np.array_equal(pos_g[:T], pos)
        emit_o, _, _ = ctrl.advance_sample(dec.logits()[:T], tau, rng, top_k=top_k, top_p=top_p)
        assert np.array_equal(emit, emit_o), (emit, emit_o)
        assert np.array_equal(dec.window(), ctrl.window())
        for key in set(int(x) for x in tok):
            assert np.array_equal(dec.pool(key), ctrl.pool(key)), key
        multi += len(emit) > 1
        P += len(emit)
        c = int(emit[-1])
    if tau <= 0.1 or top_k in (1, 2) or top_p < 1e-3:
        assert multi > 0  # candidates were accepted under sampling


@pytest.mark.parametrize("dtype", [0, 1], ids=["fp32", "bf16"])
def test_temperature_to_zero_and_back_is_greedy(dtype):
    import lossless_lookahead_decoding_gb300 as LA
    cfg, w, prompt, (W, N, G) = _setup(dtype)
    g = gpu_decoder(cfg, w, dtype, 0, 2, 0, 256).generate(prompt, 48)
    dec = gpu_decoder(cfg, w, dtype, W, N, G, 256)
    dec.set_sampling(1e-8, 5)
    assert np.array_equal(dec.generate(prompt, 48), g)
    dec.set_sampling(0.5, 6)
    dec.generate(prompt, 16)
    dec.set_sampling(0.0, 0)
    assert np.array_equal(dec.generate(prompt, 48), g)
    with pytest.raises(LA.LAError):
        dec.set_sampling(math.nan, 1)


def test_top_k_one_emits_the_largest_weight_token():
    """top_k = 1 leaves one token per row: the sampled decode is
    deterministic, the same for any uniform stream, and equals the oracle's
    top-1 ancestral decode."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg, w, prompt, (W, N, G) = _setup(0)
    a = gpu_decoder(cfg, w, 0, W, N, G, 256)
    a.set_sampling(0.9, 1, top_k=1)
    b = gpu_decoder(cfg, w, 0, W, N, G, 256)
    b.set_sampling(0.9, 12345, top_k=1)
    ta, tb = a.generate(prompt, 40), b.generate(prompt, 40)
    assert np.array_equal(ta, tb)
    assert np.array_equal(ta, O.sample_decode(O.Model(cfg, w), prompt, 40, 0.9, 3, top_k=1))
    with pytest.raises(LA.LAError):
        LA.la_set_top_k(a.ctx, -1)


def test_tiny_top_p_emits_the_largest_weight_token():
    """top_p -> 0 keeps one token per row, the largest weight: the sampled
    decode is the same for any uniform stream and equals both top_k = 1 and
    the oracle's tiny-top-p ancestral decode; out-of-range top_p fails."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg, w, prompt, (W, N, G) = _setup(1)
    a = gpu_decoder(cfg, w, 1, W, N, G, 256)
    a.set_sampling(0.9, 1, top_p=1e-7)
    b = gpu_decoder(cfg, w, 1, W, N, G, 256)
    b.set_sampling(0.9, 999, top_k=1)
    ta = a.generate(prompt, 40)
    assert np.array_equal(ta, b.generate(prompt, 40))
    for bad in (0.0, -0.5, 1.5, math.nan):
        with pytest.raises(LA.LAError):
            LA.la_set_top_p(a.ctx, bad)
    LA.la_set_top_p(a.ctx, 1.0)


@pytest.mark.parametrize("tau,top_k,top_p", [(2.0, 0, 0.9), (1.0, 6000, 0.8), (0.7, 0, 0.3), (3.0, 0, 0.999)],
                         ids=["p0.9-flat", "top6000-p0.8", "p0.3", "p0.999-flat"])
def test_7b_vocab_top_p_replays_the_oracle_rule(tau, top_k, top_p):
    """Vocabulary 32000 (a 2-layer slice at 7B widths, W=7 N=5 G=7): at high
    temperature most of the vocabulary carries weight, so the weighted radix
    select runs several passes over every token before the keys fit its
    shared-memory gather; emitted tokens, window and pool against the oracle
    rule on the GPU's logits."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["7b"].sliced(2)
    full = I.make_weights(I.MODELS["7b"], 0, bf16=True, layers=[0, 1])
    w = {k: (v[:2] if isinstance(v, list) else v) for k, v in full.items()}
    prompt = I.make_prompt("7b")
    W, N, G = 7, 5, 7
    seed = 123
    dec = gpu_decoder(cfg, w, 1, W, N, G, 640, flags=LA.LA_DEBUG_LOGITS)
    dec.set_sampling(tau, seed, top_k=top_k, top_p=top_p)
    ctrl = O.Controller(W, N, G, cfg.vocab)
    ctrl.init(prompt, seed=2)
    rng = O.Rng(seed)
    dec.prefill(prompt)
    c, P = int(prompt[-1]), len(prompt) - 1
    for _ in range(4):
        emit = dec.step()
        tok, pos, _ = ctrl.rows(c, P)
        T = len(tok)
        emit_o, _, _ = ctrl.advance_sample(dec.logits()[:T], tau, rng, top_k=top_k, top_p=top_p)
        assert np.array_equal(emit, emit_o), (emit, emit_o)
        assert np.array_equal(dec.window(), ctrl.window())
        P += len(emit)
        c = int(emit[-1])
