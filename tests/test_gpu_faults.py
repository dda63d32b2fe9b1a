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
