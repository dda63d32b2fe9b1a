"""The masked lookahead attention on its own (la_attention), through the C ABI.

* The attention micro-benchmark case: 32 heads x 128, a 2048-token bf16 KV
  cache ~ N(0,1), the W=15 N=5 G=15 query set (1 + 60 + 60 = 121 rows) with
  the combined 2D-window + verification mask; against the oracle's attention
  (fp32 on the same bf16 values), every row within rel-L2 1e-2.
* GQA with head_dim 64 at a ragged cache length, and the single-row greedy
  case.
* Bit-exactness that keeps lookahead lossless: each step row's output equals,
  bit for bit, the output of decoding that row alone (W = G = 0) after its
  visible step rows have been appended to the cache in position order --
  around the kernel's 64-position chunk and 256-position split boundaries and
  at a 31-position-wide window.
"""
import numpy as np
import pytest

import la_inputs as I
import oracle as O
from helpers import build_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()


def _rows(W, N, G, P, V=64):
    k = O.Controller(W, N, G, V)
    k.init(np.arange(V, dtype=np.int32), seed=1)
    for g in range(G):
        k.insert(3, [(g * 7 + i) % V for i in range(N - 1)])
    return k.rows(3, P)


def _run(q, kc, vc, ks, vs, H, Hkv, hd, max_seq, P, W, N, G):
    import torch
    import lossless_lookahead_decoding_gb300 as LA
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(torch.bfloat16)
    dq, dk, dv, dks, dvs = t(q), t(kc), t(vc), t(ks), t(vs)
    out = torch.zeros((q.shape[0], H * hd), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    rc = LA.la_attention(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dks.data_ptr(), dvs.data_ptr(),
                         out.data_ptr(), H, Hkv, hd, max_seq, P, W, N, G, st.cuda_stream)
    assert rc == 0, rc
    return out.float().cpu().numpy().reshape(q.shape[0], H, hd)


def _case(H, Hkv, hd, P, W, N, G, seed):
    g = np.random.default_rng(seed)
    max_seq = P + W + N + 32
    f = lambda *s: I.bf16_round(g.standard_normal(s, dtype=np.float32))
    T = 1 + (W + G) * (N - 1)
    kc, vc = np.zeros((Hkv, max_seq, hd), np.float32), np.zeros((Hkv, max_seq, hd), np.float32)
    kc[:, :P], vc[:, :P] = f(Hkv, P, hd), f(Hkv, P, hd)
    return f(T, H, hd), kc, vc, f(T, Hkv, hd), f(T, Hkv, hd), max_seq


def _check_against_oracle(H, Hkv, hd, P, W, N, G, seed, tol=1e-2):
    q, kc, vc, ks, vs, max_seq = _case(H, Hkv, hd, P, W, N, G, seed)
    tok, pos, vis = _rows(W, N, G, P)
    ref = O.attention(q, kc, vc, ks, vs, vis, pos, P)
    got = _run(q, kc, vc, ks, vs, H, Hkv, hd, max_seq, P, W, N, G)
    err = np.linalg.norm((got - ref).reshape(len(q), -1), axis=1) / np.linalg.norm(ref.reshape(len(q), -1), axis=1)
    assert err.max() <= tol, err.max()
    return q, kc, vc, ks, vs, max_seq, pos, vis, got


def test_microbench_case_against_oracle():
    """32 x 128 heads, 2048 cached tokens, W=15 N=5 G=15 (121 rows)."""
    inp = I.attention_bench_inputs()
    H, hd, P, W, N, G = 32, 128, 2048, 15, 5, 15
    max_seq = P + 64
    kc = np.zeros((H, max_seq, hd), np.float32)
    vc = np.zeros((H, max_seq, hd), np.float32)
    kc[:, :P], vc[:, :P] = inp["k_cache"], inp["v_cache"]
    tok, pos, vis = _rows(W, N, G, P)
    assert len(tok) == 121
    ref = O.attention(inp["q"], kc, vc, inp["k_step"], inp["v_step"], vis, pos, P)
    got = _run(inp["q"], kc, vc, inp["k_step"], inp["v_step"], H, H, hd, max_seq, P, W, N, G)
    err = np.linalg.norm((got - ref).reshape(121, -1), axis=1) / np.linalg.norm(ref.reshape(121, -1), axis=1)
    assert err.max() <= 1e-2, err.max()


@pytest.mark.parametrize("H,Hkv,hd,P,W,N,G", [(32, 8, 64, 1000, 4, 3, 4), (8, 8, 128, 777, 0, 2, 0),
                                               (4, 2, 128, 63, 7, 5, 7), (4, 4, 64, 0, 3, 4, 2),
                                               # short caches, and caches ending next to chunk and split
                                               # boundaries
                                               (4, 4, 128, 10, 15, 5, 15), (4, 4, 128, 40, 15, 5, 15),
                                               (8, 2, 128, 256 + 31, 7, 5, 7), (4, 1, 64, 129, 5, 3, 5),
                                               # windows 31 positions wide: W + N - 2 = 31
                                               (8, 8, 128, 300, 28, 5, 2), (4, 4, 128, 517, 30, 3, 30)])
def test_shapes_against_oracle(H, Hkv, hd, P, W, N, G):
    _check_against_oracle(H, Hkv, hd, P, W, N, G, seed=H + P)


@pytest.mark.parametrize("P", [0, 17, 127, 128, 143, 250, 319, 1023])
def test_rows_equal_their_greedy_decoding_bitwise(P):
    H, Hkv, hd, W, N, G = 4, 2, 128, 7, 5, 7
    q, kc, vc, ks, vs, max_seq, pos, vis, got = _check_against_oracle(H, Hkv, hd, P, W, N, G, seed=P)
    T = len(q)
    for r in [0, 1, 7, 8, 1 + 3 * W + 6, 1 + W * (N - 1), T - 1, T - 2]:
        seen = sorted((pos[c], c) for c in range(T) if vis[r, c] and c != r)
        kc2, vc2 = kc.copy(), vc.copy()
        for p, c in seen:
            kc2[:, p], vc2[:, p] = ks[c], vs[c]
        alone = _run(q[r:r + 1], kc2, vc2, ks[r:r + 1], vs[r:r + 1], H, Hkv, hd, max_seq, int(pos[r]), 0, 2, 0)
        assert np.array_equal(alone[0], got[r]), r


@pytest.mark.parametrize("P", [33, 300, 641])
def test_widest_window_rows_equal_their_greedy_decoding_bitwise(P):
    """W + N - 2 = 31: the lookahead rows reach 31 positions past the
    cache."""
    H, Hkv, hd, W, N, G = 4, 4, 64, 28, 5, 2
    q, kc, vc, ks, vs, max_seq, pos, vis, got = _check_against_oracle(H, Hkv, hd, P, W, N, G, seed=P + 5)
    T = len(q)
    for r in [0, 1, 28, 29, 1 + 3 * W + W - 1, T - 1]:
        seen = sorted((pos[c], c) for c in range(T) if vis[r, c] and c != r)
        kc2, vc2 = kc.copy(), vc.copy()
        for p, c in seen:
            kc2[:, p], vc2[:, p] = ks[c], vs[c]
        alone = _run(q[r:r + 1], kc2, vc2, ks[r:r + 1], vs[r:r + 1], H, Hkv, hd, max_seq, int(pos[r]), 0, 2, 0)
        assert np.array_equal(alone[0], got[r]), r
