"""la_attention_noalloc: the attention op for callers that cannot allocate
device memory, with its scratch in the library's fixed device array.

Called through the C ABI twice in a row with different inputs (the array
keeps the previous call's contents), each result compared with
la_attention's (which allocates its own scratch) on the same inputs; and a
configuration larger than the fixed array must be refused.  Collected last
so that a failure here leaves every other test already run.
"""
import numpy as np
import pytest

from helpers import build_lib

pytestmark = pytest.mark.gpu


def _inputs(seed, H, Hkv, hd, P, T, max_seq):
    import torch
    g = torch.Generator(device="cpu").manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16).cuda()
    kc = torch.zeros((Hkv, max_seq, hd), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kc[:, :P], vc[:, :P] = r(Hkv, P, hd), r(Hkv, P, hd)
    return r(T, H, hd), kc, vc, r(T, Hkv, hd), r(T, Hkv, hd)


def test_noalloc_matches_allocating_entry_point():
    import torch
    build_lib()
    import lossless_lookahead_decoding_gb300 as LA
    st = torch.cuda.Stream()
    H, Hkv, hd, W, N, G = 32, 32, 128, 15, 5, 15
    T = 1 + (W + G) * (N - 1)
    for seed, P in ((11, 700), (12, 389)):
        max_seq = 768
        q, kc, vc, ks, vs = _inputs(seed, H, Hkv, hd, P, T, max_seq)
        ref = torch.zeros((T, H * hd), dtype=torch.bfloat16, device="cuda")
        got = torch.full((T, H * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        args = (q.data_ptr(), kc.data_ptr(), vc.data_ptr(), ks.data_ptr(), vs.data_ptr())
        assert LA.la_attention(*args, ref.data_ptr(), H, Hkv, hd, max_seq, P, W, N, G, st.cuda_stream) == 0
        assert LA.la_attention_noalloc(*args, got.data_ptr(), H, Hkv, hd, max_seq, P, W, N, G, st.cuda_stream) == 0
        torch.cuda.synchronize()
        a, b = got.float().cpu().numpy(), ref.float().cpu().numpy()
        assert np.isfinite(a).all()
        err = np.linalg.norm(a - b, axis=1) / np.linalg.norm(b, axis=1)
        assert err.max() <= 1e-2  # the bf16 tolerance of the other parity tests
        assert np.array_equal(a, b)  # same kernels, same inputs: in fact bit-identical


def test_noalloc_refuses_oversized_scratch():
    import torch
    build_lib()
    import lossless_lookahead_decoding_gb300 as LA
    H, hd, max_seq = 64, 128, 4096  # 64 heads x 32 splits of partials: > 16 MiB
    q, kc, vc, ks, vs = _inputs(3, H, H, hd, 100, 1, max_seq)
    out = torch.zeros((1, H * hd), dtype=torch.bfloat16, device="cuda")
    rc = LA.la_attention_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), ks.data_ptr(), vs.data_ptr(),
                                 out.data_ptr(), H, H, hd, max_seq, 100, 0, 2, 0, 0)
    assert rc == LA.LA_ERR_CAPACITY
