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


@pytest.mark.parametrize("dtype,flags", [(0, 0), (1, 0), (1, 64), (1, 32)],
                         ids=["fp32", "bf16", "bf16-diagonal", "bf16-attntc"])
def test_sampled_steps_replay_the_oracle_rule(dtype, flags):
    import lossless_lookahead_decoding_gb300 as LA
    cfg, w, prompt, (W, N, G) = _setup(dtype)
    tau, seed = 0.05, 77
    dec = gpu_decoder(cfg, w, dtype, W, N, G, 256, flags=flags | LA.LA_DEBUG_LOGITS)
    dec.set_sampling(tau, seed)
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
        emit_o, _, _ = ctrl.advance_sample(dec.logits()[:T], tau, rng)
        assert np.array_equal(emit, emit_o), (emit, emit_o)
        assert np.array_equal(dec.window(), ctrl.window())
        for key in set(int(x) for x in tok):
            assert np.array_equal(dec.pool(key), ctrl.pool(key)), key
        multi += len(emit) > 1
        P += len(emit)
        c = int(emit[-1])
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
