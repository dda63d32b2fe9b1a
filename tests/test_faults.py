"""Host-side fault injection (LA_FAULT), on the host only: la_create fails as
if the workspace allocation failed or the arguments were refused, before any
CUDA call is made, so these run without a GPU.  (The step-time injections,
timeout@K and capacity@K, are exercised by tests/test_gpu_faults.py.)"""
import os

import pytest

from helpers import build_lib


def _desc(LA):
    return LA.la_model_desc(n_layers=2, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=688, vocab=1024,
                            max_seq=256, rms_eps=1e-5, rope_theta=1e4, dtype=LA.LA_BF16, emb=1, layer_w=None,
                            final_norm=1, lm_head=1, stream=None)


@pytest.mark.parametrize("fault,code", [("alloc", -2), ("badarg", -1)])
def test_create_failures_are_injected_on_the_host(fault, code, monkeypatch):
    import ctypes as C
    build_lib()
    import lossless_lookahead_decoding_gb300 as LA
    ptrs = (C.c_void_p * 18)(*([1] * 18))
    d = _desc(LA)
    d.layer_w = C.cast(ptrs, C.c_void_p).value
    monkeypatch.setenv("LA_FAULT", fault)
    with pytest.raises(LA.LAError) as e:
        LA.la_create(d, 4, 3, 4)
    assert e.value.code == code
    monkeypatch.delenv("LA_FAULT")
    assert os.environ.get("LA_FAULT") is None
