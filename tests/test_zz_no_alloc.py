"""la_attention_noalloc: the attention op for callers that cannot allocate
device memory, with its scratch in the library's fixed device array.

Called through the C ABI twice in a row with different inputs (the array
keeps the previous call's contents), each result compared with
la_attention's (which allocates its own scratch) on the same inputs; a
configuration larger than the fixed array must be refused, and the two
configurations on either side of the array's size behave accordingly.
Collected last
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


def _need(H, hd, max_seq):
    """The documented scratch size for plain greedy rows (W = G = 0, N = 2:
    one row group, largest offset 0)."""
    c256 = lambda x: (x + 255) // 256 * 256
    state = 112  # the decode-state word: 8 ints, 2 x 8 ints, 2 x 8 bytes
    return c256((5 * 128 + 1 + 1 * 1) * 4) + c256(state) + H * -(-max_seq // 256) * 128 * (hd + 4) * 4


def test_noalloc_refuses_oversized_scratch():
    import torch
    build_lib()
    import lossless_lookahead_decoding_gb300 as LA
    H, hd, max_seq = 64, 128, 4096  # 64 heads x 16 splits of 256 positions: 17.3 MB of partials
    assert _need(H, hd, max_seq) > 16 << 20
    q, kc, vc, ks, vs = _inputs(3, H, H, hd, 100, 1, max_seq)
    out = torch.zeros((1, H * hd), dtype=torch.bfloat16, device="cuda")
    rc = LA.la_attention_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), ks.data_ptr(), vs.data_ptr(),
                                 out.data_ptr(), H, H, hd, max_seq, 100, 0, 2, 0, 0)
    assert rc == LA.LA_ERR_CAPACITY


@pytest.mark.parametrize("H,fits", [(62, True), (63, False)])
def test_noalloc_at_the_array_boundary(H, fits):
    """max_seq 1024 (4 splits), head_dim 128: 62 heads need 16 763 904 bytes,
    13 KB under the 16 MiB array, and run (equal to la_attention); 63 heads
    need 17 034 240 and are refused."""
    import torch
    build_lib()
    import lossless_lookahead_decoding_gb300 as LA
    hd, max_seq, P = 128, 1024, 900
    assert (_need(H, hd, max_seq) <= 16 << 20) == fits
    q, kc, vc, ks, vs = _inputs(5 + H, H, H, hd, P, 1, max_seq)
    args = (q.data_ptr(), kc.data_ptr(), vc.data_ptr(), ks.data_ptr(), vs.data_ptr())
    got = torch.full((1, H * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    rc = LA.la_attention_noalloc(*args, got.data_ptr(), H, H, hd, max_seq, P, 0, 2, 0, st.cuda_stream)
    if not fits:
        assert rc == LA.LA_ERR_CAPACITY
        return
    assert rc == 0
    ref = torch.zeros((1, H * hd), dtype=torch.bfloat16, device="cuda")
    assert LA.la_attention(*args, ref.data_ptr(), H, H, hd, max_seq, P, 0, 2, 0, st.cuda_stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
