"""GPU n-gram pool (hash table) vs the oracle's pool, bit for bit: the pool
micro-benchmark case (4096 keys x 15 4-grams over a 32000-token vocabulary,
Zipf(1.1) tokens, inserts with eviction and duplicates), through the C ABI."""
import numpy as np
import pytest

import la_inputs as I
import oracle as O
from helpers import build_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()


def _oracle_pool(keys, grams, N, G, V):
    k = O.Controller(0, N, G, V)
    for key, gram in zip(keys.tolist(), grams):
        k.insert(key, gram)
    return k


@pytest.mark.parametrize("n_keys,per_key,G", [(4096, 20, 15), (300, 3, 4), (1, 40, 7)])
def test_bulk_insert_and_lookup(n_keys, per_key, G):
    import torch
    import lossless_lookahead_decoding_gb300 as LA
    N, V = 5, 32000
    keys, grams = I.pool_bench_inserts(n_keys, per_key, V, N - 1)
    # duplicates: re-insert a slice (no-ops unless evicted meanwhile)
    keys = np.concatenate([keys, keys[:50]])
    grams = np.concatenate([grams, grams[:50]])
    ref = _oracle_pool(keys, grams, N, G, V)
    pool = LA.la_pool_create(2 * n_keys + 64, N, G)
    dk = torch.from_numpy(keys).cuda()
    dg = torch.from_numpy(np.ascontiguousarray(grams)).cuda()
    assert LA.la_pool_insert(pool, dk.data_ptr(), dg.data_ptr(), len(keys)) == 0
    uniq = np.unique(keys)
    assert LA.la_pool_size(pool) == len(uniq)
    q = np.concatenate([uniq, np.array([31999, 0, 12345], np.int32)])
    q = q[~np.isin(q, uniq) | (np.arange(len(q)) < len(uniq))]
    dq = torch.from_numpy(q).cuda()
    out = torch.empty((len(q), G, N - 1), dtype=torch.int32, device="cuda")
    cnt = torch.empty(len(q), dtype=torch.int32, device="cuda")
    assert LA.la_pool_lookup(pool, dq.data_ptr(), len(q), out.data_ptr(), cnt.data_ptr()) == 0
    torch.cuda.synchronize()
    out, cnt = out.cpu().numpy(), cnt.cpu().numpy()
    for i, key in enumerate(q.tolist()):
        want = ref.pool(key)
        assert cnt[i] == len(want)
        assert np.array_equal(out[i, :cnt[i]], want)
        assert (out[i, cnt[i]:] == -1).all()
    LA.la_pool_destroy(pool)


def test_pool_capacity_error():
    import torch
    import lossless_lookahead_decoding_gb300 as LA
    pool = LA.la_pool_create(64, 3, 2)
    keys = torch.arange(100, dtype=torch.int32, device="cuda")
    grams = torch.zeros((100, 2), dtype=torch.int32, device="cuda")
    assert LA.la_pool_insert(pool, keys.data_ptr(), grams.data_ptr(), 100) == LA.LA_ERR_CAPACITY
    LA.la_pool_destroy(pool)


def test_negative_keys_are_refused_and_absent():
    """-1 marks empty slots, so a negative key is refused by insert
    (LA_ERR_ARG; the other inserts of the batch are made) and looked up as
    absent; a later insert succeeds again (the status is per call)."""
    import torch
    import lossless_lookahead_decoding_gb300 as LA
    N, G = 3, 2
    pool = LA.la_pool_create(64, N, G)
    keys = torch.tensor([5, -1, 7, -3], dtype=torch.int32, device="cuda")
    grams = torch.tensor([[1, 2], [3, 4], [5, 6], [7, 8]], dtype=torch.int32, device="cuda")
    assert LA.la_pool_insert(pool, keys.data_ptr(), grams.data_ptr(), 4) == LA.LA_ERR_ARG
    assert LA.la_pool_size(pool) == 2
    q = torch.tensor([5, 7, -1, -3, 9], dtype=torch.int32, device="cuda")
    out = torch.empty((5, G, N - 1), dtype=torch.int32, device="cuda")
    cnt = torch.empty(5, dtype=torch.int32, device="cuda")
    assert LA.la_pool_lookup(pool, q.data_ptr(), 5, out.data_ptr(), cnt.data_ptr()) == 0
    torch.cuda.synchronize()
    assert cnt.cpu().tolist() == [1, 1, 0, 0, 0]
    assert out[0, 0].cpu().tolist() == [1, 2] and out[1, 0].cpu().tolist() == [5, 6]
    assert (out[2:].cpu() == -1).all()
    ok = torch.tensor([9], dtype=torch.int32, device="cuda")
    assert LA.la_pool_insert(pool, ok.data_ptr(), grams.data_ptr(), 1) == LA.LA_OK
    LA.la_pool_destroy(pool)
