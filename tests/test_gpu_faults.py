"""Step-time fault injection from the host (LA_FAULT=timeout@K|capacity@K):
no kernel is made to fail or wait.  timeout@K: the host writes the status a
bounded device wait sets when it gives up, so the K-th step returns
LA_ERR_TIMEOUT, the context refuses steps until la_prefill, and after it the
decode is the plain greedy one again.  capacity@K: the K-th step reports a
full cache and the next step carries on."""
import numpy as np
import pytest

import la_inputs as I
from helpers import build_lib, gpu_decoder

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()


def _setup():
    cfg = I.MODELS["tiny"]
    w = I.make_weights(cfg, 0, bf16=True)
    prompt = I.make_prompt("tiny")
    g = gpu_decoder(cfg, w, 1, 0, 2, 0, 256).generate(prompt, 24)
    return cfg, w, prompt, g


def test_injected_timeout_and_recovery(monkeypatch):
    import lossless_lookahead_decoding_gb300 as LA
    cfg, w, prompt, g = _setup()
    monkeypatch.setenv("LA_FAULT", "timeout@3")
    dec = gpu_decoder(cfg, w, 1, 4, 3, 4, 256)
    monkeypatch.delenv("LA_FAULT")
    dec.prefill(prompt)
    out = list(dec.step()) + list(dec.step())
    with pytest.raises(LA.LAError) as e:
        dec.step()
    assert e.value.code == LA.LA_ERR_TIMEOUT
    with pytest.raises(LA.LAError) as e:
        dec.step()
    assert e.value.code == LA.LA_ERR_STATE
    assert np.array_equal(out, g[:len(out)])
    # after a prefill the context decodes again (the injection was for step 3)
    toks = dec.generate(prompt, 24)
    assert np.array_equal(toks, g)
    dec.close()


def test_injected_capacity_then_continue(monkeypatch):
    import lossless_lookahead_decoding_gb300 as LA
    cfg, w, prompt, g = _setup()
    monkeypatch.setenv("LA_FAULT", "capacity@2")
    dec = gpu_decoder(cfg, w, 1, 4, 3, 4, 256)
    monkeypatch.delenv("LA_FAULT")
    dec.prefill(prompt)
    out = list(dec.step())
    with pytest.raises(LA.LAError) as e:
        dec.step()
    assert e.value.code == LA.LA_ERR_CAPACITY
    while len(out) < 24:
        out += list(dec.step())
    assert np.array_equal(out[:24], g)
    dec.close()


def test_injected_timeout_in_a_batched_context(monkeypatch):
    """timeout@K on a batched context: the K-th batched step returns
    LA_ERR_TIMEOUT, every sequence then needs its prefill again, and after
    it each sequence decodes as a batch-1 greedy context does."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg, w, prompt, g = _setup()
    dw = LA.device_weights(cfg, w, LA.LA_BF16)
    monkeypatch.setenv("LA_FAULT", "timeout@2")
    dec = LA.Decoder(cfg, dw, LA.LA_BF16, 4, 3, 4, 256, batch=2)
    monkeypatch.delenv("LA_FAULT")
    p2 = prompt[:20]
    dec.prefill_seq(0, prompt)
    dec.prefill_seq(1, p2)
    dec.step_batch()
    with pytest.raises(LA.LAError) as e:
        dec.step_batch()
    assert e.value.code == LA.LA_ERR_TIMEOUT
    with pytest.raises(LA.LAError) as e:
        dec.step_batch()
    assert e.value.code == LA.LA_ERR_STATE
    dec.prefill_seq(0, prompt)
    with pytest.raises(LA.LAError) as e:  # sequence 1 still needs its prefill
        dec.step_batch()
    assert e.value.code == LA.LA_ERR_STATE
    dec.prefill_seq(1, p2)
    outs = [[], []]
    while min(len(o) for o in outs) < 24:
        for b, t in enumerate(dec.step_batch()):
            outs[b].extend(t.tolist())
    g2 = gpu_decoder(cfg, w, 1, 0, 2, 0, 256).generate(p2, 24)
    assert np.array_equal(np.array(outs[0][:24], np.int32), g)
    assert np.array_equal(np.array(outs[1][:24], np.int32), g2)


def test_profiled_batched_context_keeps_the_output():
    """LA_PROFILE | LA_NO_GRAPH on a batched context: the same tokens as the
    graph-launched batched context, and the profile's kernel classes."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg, w, prompt, g = _setup()
    dw = LA.device_weights(cfg, w, LA.LA_BF16)
    prompts = [prompt, prompt[:24]]
    a = LA.Decoder(cfg, dw, LA.LA_BF16, 4, 3, 4, 256, batch=2).generate_batch(prompts, 24)
    dec = LA.Decoder(cfg, dw, LA.LA_BF16, 4, 3, 4, 256, flags=LA.LA_PROFILE | LA.LA_NO_GRAPH, batch=2)
    b = dec.generate_batch(prompts, 24)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    prof = dec.profile()
    for cls in ("gemm_qkv", "attention", "control"):
        assert prof[cls]["launches"] > 0, cls
