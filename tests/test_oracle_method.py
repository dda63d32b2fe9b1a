"""Pins of the oracle's lookahead decoding against what the pages and the
mathematics fix (not against the oracle itself):

* losslessness: lookahead output == greedy output token for token (the
  summary's claim that the output distribution stays exactly the same);
* the step shape against the pages' printed FLOPs overheads (Key points);
* gap-free causal visibility of every row of the combined mask, and per-row
  equivalence of the masked forward with the plain causal forward;
* verification: brute force over all candidate sets on a tiny vocabulary with
  a bigram "model" whose greedy continuation is known in closed form;
* the pool: replay against a list-of-tuples simulator;
* reductions: W=G=0 is greedy, G=0 emits one token per step, W=0 with a
  prompt-seeded pool only ever holds prompt n-grams;
* splitmix64 known-answer outputs, the window initialisation (reading R1)
  and the sampling uniforms written out from them;
* the "diagonal levels" mask reading R3' (each level one Jacobi iterate over
  the same positions, n-grams along diagonals): the same visibility,
  per-row, pool-replay and losslessness pins, plus a bigram model on which
  every harvested n-gram must be a chain of the model's own predictions --
  true of the harvest direction that matches the window update (columns
  under R3, diagonals under R3') and false of the other.
"""
import itertools
import os

import numpy as np
import pytest

import la_inputs as I
import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
SMALL = I.ModelConfig("small-gqa", 2, 64, 4, 2, 16, 96, 50)
MICRO = I.ModelConfig("micro", 1, 32, 2, 1, 16, 48, 24)


def _golden(name):
    rows = []
    for line in open(os.path.join(GOLD, name)):
        line = line.split("#")[0].split()
        if line:
            rows.append(line)
    return rows


def test_splitmix64_known_answers():
    for row in _golden("splitmix64_kat.txt"):
        seed, vals = int(row[0]), [int(v) for v in row[1:]]
        assert O.splitmix64_stream(seed, len(vals)) == vals


def _kat_stream(seed):
    for row in _golden("splitmix64_kat.txt"):
        if int(row[0]) == seed:
            return [int(v) for v in row[1:]]
    raise KeyError(seed)


@pytest.mark.parametrize("W,N", [(5, 2), (2, 3), (1, 6), (1, 2)])
def test_window_init_from_the_splitmix64_stream(W, N):
    """Reading R1, written out from the golden known answers (not from the
    oracle's generator): win[l][j] = prompt[x_k mod len], x_k the k-th output
    of the stream seeded with the window seed, k = l*W + j (level-major).  The
    prompt's tokens are distinct, so a swapped l/j order, an off-by-one in the
    index or a wrong modulus all change the window."""
    xs = _kat_stream(1234567)
    assert len(xs) >= W * (N - 1)
    prompt = (1000 + 7 * np.arange(97)).astype(np.int32)
    k = O.Controller(W, N, 0, 2000)
    k.init(prompt, seed=1234567)
    expect = np.array([prompt[x % len(prompt)] for x in xs[:W * (N - 1)]], np.int32).reshape(N - 1, W)
    assert np.array_equal(k.window(), expect)
    # a one-token prompt fills the whole window with that token
    k.init(np.array([42], np.int32), seed=1234567)
    assert (k.window() == 42).all()


def test_uniform_is_the_top_24_bits_of_the_stream():
    """The sampling verification's uniforms: (x >> 40) / 2^24 for the stream's
    outputs x, written out from the golden known answers."""
    xs = _kat_stream(1234567)
    r = O.Rng(1234567)
    got = [r.uniform() for _ in xs]
    assert got == [(x >> 40) / 2.0 ** 24 for x in xs]
    assert all(0.0 <= u < 1.0 for u in got)


@pytest.mark.parametrize("row", _golden("page_settings.txt"), ids=lambda r: r[0])
def test_step_rows_match_pages_flops_overhead(row):
    """With a full pool, a step has 1 + (W+G)(N-1) rows; at G = W the extra
    rows are 2W(N-1), the pages' 120x / 80x / 56x per-step FLOPs overhead."""
    W, N, G, extra = map(int, row[1:])
    V = 40
    k = O.Controller(W, N, G, V)
    k.init(np.arange(V, dtype=np.int32), seed=2)
    for g in range(G):
        k.insert(5, [g + 1] * (N - 1))
    tok, pos, vis = k.rows(5, 100)
    assert len(tok) - 1 == extra
    assert len(tok) == k.Tmax


def test_attention_microbench_row_count():
    """The 1 + 60 + 60 = 121 query rows of the W=15 N=5 G=15 attention case."""
    k = O.Controller(15, 5, 15, 64)
    assert k.Tmax == 121


def _check_visibility(tok, pos, vis, P, W, N, G, variant=0):
    T = len(tok)
    for r in range(T):
        seen = sorted(pos[s] for s in range(T) if vis[r, s])
        assert seen == list(range(P, pos[r] + 1)), (r, seen)
    if variant == 0:
        # each lookahead column is a run of consecutive positions, level by level
        for j in range(W):
            ps = [pos[1 + l * W + j] for l in range(N - 1)]
            assert ps == list(range(P + 1 + j, P + 1 + j + N - 1))
    else:
        # each level covers P+1..P+W and sees only itself (and row 0)
        for l in range(N - 1):
            lv = [1 + l * W + j for j in range(W)]
            assert [pos[r] for r in lv] == list(range(P + 1, P + 1 + W))
            for j, r in enumerate(lv):
                assert sorted(np.flatnonzero(vis[r]).tolist()) == [0] + lv[:j + 1]


@pytest.mark.parametrize("variant", [0, O.DIAGONAL], ids=["R3", "diagonal"])
def test_mask_brute_force_gap_free(variant):
    for W, N, G in itertools.product(range(5), range(2, 5), range(4)):
        k = O.Controller(W, N, G, 32, variant=variant)
        k.init(np.arange(32, dtype=np.int32), seed=W * 100 + N * 10 + G)
        for g in range(G):
            k.insert(3, [(g + 7 * i) % 32 for i in range(N - 1)])
        tok, pos, vis = k.rows(3, 11)
        assert len(tok) == 1 + (W + G) * (N - 1)
        _check_visibility(tok, pos, vis, 11, W, N, G, variant)


@pytest.mark.parametrize("variant", [0, O.DIAGONAL], ids=["R3", "diagonal"])
@pytest.mark.parametrize("W,N,G", [(4, 3, 4), (2, 4, 3), (3, 2, 2), (0, 3, 2), (3, 3, 0)])
def test_masked_rows_equal_plain_causal_forward(W, N, G, variant):
    """Row r of the combined step equals, bit for bit, the plain causal forward
    of the token sequence row r sees (its visible positions in order)."""
    cfg = SMALL
    m = O.Model(cfg, I.make_weights(cfg, 0))
    prompt = I.random_prompt(9, cfg.vocab, 11)
    P = len(prompt) - 1
    k = O.Controller(W, N, G, cfg.vocab, variant=variant)
    k.init(prompt, seed=5)
    c = int(prompt[-1])
    g = np.random.default_rng(2)
    for _ in range(G):
        k.insert(c, g.integers(0, cfg.vocab, N - 1))
    tok, pos, vis = k.rows(c, P)
    s = O.Seq(m, 64)
    s.prefill(prompt[:-1])
    lg, amax = s.step(P, tok, pos, vis)
    for r in range(len(tok)):
        order = sorted((pos[t], t) for t in range(len(tok)) if vis[r, t])
        seq = np.concatenate([prompt[:-1], [tok[t] for _, t in order]]).astype(np.int32)
        ref = O.Seq(m, 64)
        ref.prefill(seq[:-1])
        lr, ar = ref.step(len(seq) - 1, seq[-1:], [len(seq) - 1], [[1]])
        assert np.array_equal(lr[0], lg[r]), r
        assert ar[0] == amax[r]


def test_verify_brute_force_bigram():
    """A bigram model f: every row's argmax is f(its token), so the greedy
    continuation of c is s1 = f(c), s2 = f(s1), ...  For every ordered set of
    candidate 2-grams the step must emit s1..s(m+1), m = the longest common
    prefix of a candidate with (s1, s2), first such candidate chosen."""
    V, N = 3, 3
    grams = list(itertools.product(range(V), repeat=N - 1))
    c = 0
    for table in itertools.product(range(V), repeat=V):
        f = lambda t: table[t]
        greedy = [f(c)]
        for _ in range(N - 1):
            greedy.append(f(greedy[-1]))
        for G in range(0, 4):
            for cands in itertools.permutations(grams, G):
                k = O.Controller(0, N, G, V)
                k.init([c], seed=1)
                for cand in cands:
                    k.insert(c, cand)
                tok, pos, vis = k.rows(c, 4)
                emit, rows, gstar = k.advance([f(t) for t in tok])
                lcp = [next((i for i in range(N - 1) if cand[i] != greedy[i]), N - 1) for cand in cands]
                m = max(lcp) if lcp else 0
                assert list(emit) == greedy[:m + 1]
                assert gstar == (lcp.index(m) if lcp else -1)
                assert 1 <= len(emit) <= N


def _sim_insert(pool, key, val, G):
    if G == 0:
        return
    lst = pool.setdefault(key, [])
    if val in lst:
        return
    if len(lst) == G:
        lst.pop(0)
    lst.append(val)


@pytest.mark.parametrize("variant", [0, O.DIAGONAL], ids=["R3", "diagonal"])
@pytest.mark.parametrize("W,N,G", [(4, 3, 4), (5, 4, 2), (3, 2, 3), (6, 5, 1), (2, 3, 0), (2, 4, 3)])
def test_pool_replay_against_list_simulator(W, N, G, variant):
    V = 12
    g = np.random.default_rng(W * 31 + N * 7 + G)
    prompt = g.integers(0, V, 20).astype(np.int32)
    k = O.Controller(W, N, G, V, variant=variant)
    k.init(prompt, seed=9, preseed=True)
    pool = {}
    for i in range(len(prompt) - N + 1):
        _sim_insert(pool, int(prompt[i]), tuple(int(t) for t in prompt[i + 1:i + N]), G)
    win = k.window().tolist()
    c = int(prompt[-1])
    for step in range(60):
        tok, pos, vis = k.rows(c, 19 + step)
        amax = g.integers(0, V, len(tok))
        emit, rows, gstar = k.advance(amax)
        out = [int(amax[1 + (N - 2) * W + j]) for j in range(W)]  # the last level's rows
        if variant == 0:
            for j in range(W):
                _sim_insert(pool, win[0][j], tuple(win[l][j] for l in range(1, N - 1)) + (out[j],), G)
            last = out
        else:
            # an n-gram steps one column right per level; only those that stay
            # inside the window are harvested
            for j in range(W - (N - 2)):
                _sim_insert(pool, win[0][j], tuple(win[l][j + l] for l in range(1, N - 1)) + (out[j + N - 2],), G)
            last = [int(amax[0])] + out[:W - 1]  # Jacobi update: column j from column j-1
        win = win[1:] + [last]
        assert k.window().tolist() == win
        for key in range(V):
            got = [tuple(int(x) for x in r) for r in k.pool(key)]
            assert got == pool.get(key, [])
            assert len(got) <= G and len(set(got)) == len(got)
        c = int(emit[-1])


@pytest.mark.parametrize("variant", [0, O.DIAGONAL], ids=["R3", "diagonal"])
@pytest.mark.parametrize("W,N", [(6, 4), (5, 2), (4, 5)])
def test_harvested_ngrams_are_the_models_own_chains(W, N, variant):
    """Bigram model f (every row's argmax is f of its own token).  Once the
    window's levels have been replaced by model outputs (N-2 updates), each
    level follows from the one before it by the window update, so every
    n-gram harvested after that is a chain (x, f(x), f(f(x)), ...) -- along
    columns under R3, along diagonals under R3'.  Harvesting the other
    direction (or with an off-by-one column) puts non-chains into the pool.
    Under R3' the Jacobi update puts the current token's own continuation
    into column 0, so its chain reaches the pool and later steps emit N
    tokens."""
    V = 23
    table = np.random.default_rng(5).permutation(V)  # a permutation: chains never collapse
    f = lambda t: int(table[t])
    G = 4
    k = O.Controller(W, N, G, V, variant=variant)
    prompt = np.random.default_rng(6).integers(0, V, 17).astype(np.int32)
    k.init(prompt, seed=3)
    c, P = int(prompt[-1]), len(prompt) - 1
    full = 0
    snap = lambda: {(key, tuple(v.tolist())) for key in range(V) for v in k.pool(key)}
    new_total = 0
    for step in range(40):
        tok, pos, vis = k.rows(c, P)
        before = snap()
        emit, rows, gstar = k.advance([f(t) for t in tok])
        # lossless on this model: the emitted tokens are c's greedy chain
        chain = [f(c)]
        while len(chain) < len(emit):
            chain.append(f(chain[-1]))
        assert emit.tolist() == chain
        if step >= N - 2:  # the harvest reads the window after `step` updates
            for key, v in snap() - before:
                x = [key, *v]
                assert all(x[i + 1] == f(x[i]) for i in range(N - 1)), (step, x)
                new_total += 1
            full += len(emit) == N
        P += len(emit)
        c = int(emit[-1])
    assert new_total > 0
    if variant == O.DIAGONAL:
        assert full > 0


def _lossless(cfg, bf16, W, N, G, seed, n_new, prompt, preseed=False, variant=0):
    m = O.Model(cfg, I.make_weights(cfg, 0, bf16=bf16))
    g = O.greedy(m, prompt, n_new)
    la, steps, hist = O.lookahead(m, prompt, W, N, G, n_new, seed=seed, preseed=preseed, variant=variant)
    assert np.array_equal(la, g), (W, N, G, seed)
    assert hist.sum() == steps and hist[0] == 0
    assert (hist[N + 1:] == 0).all() if len(hist) > N + 1 else True
    return steps, hist


@pytest.mark.parametrize("variant", [0, O.DIAGONAL], ids=["R3", "diagonal"])
@pytest.mark.parametrize("bf16", [False, True])
def test_lossless_tiny_workload(bf16, variant):
    W, N, G = I.LOOKAHEAD["tiny"]
    steps, hist = _lossless(I.MODELS["tiny"], bf16, W, N, G, 2, 64, I.make_prompt("tiny"), variant=variant)
    assert steps < 64  # some candidate was accepted on the planted-span prompt


@pytest.mark.parametrize("W,G", [(28, 2), (25, 5), (20, 10), (15, 15), (10, 20), (5, 25), (2, 28)])
def test_lossless_branch_balance_at_121_rows(W, G):
    """The branch-balance splits of the sweep (W + G = 30, N = 5, T = 121 rows,
    the 7B step's row count) on the tiny model: lossless at every split."""
    steps, hist = _lossless(I.MODELS["tiny"], False, W, 5, G, 2, 64, I.make_prompt("tiny"))
    assert 1 + (W + G) * 4 == 121 and steps < 64


@pytest.mark.parametrize("variant", [0, O.DIAGONAL], ids=["R3", "diagonal"])
def test_lossless_random_cases(variant):
    g = np.random.default_rng(123 + variant)
    for case in range(40):
        W, N, G = int(g.integers(0, 6)), int(g.integers(2, 6)), int(g.integers(0, 6))
        prompt = g.integers(0, MICRO.vocab, int(g.integers(1, 12))).astype(np.int32)
        _lossless(MICRO, bool(case % 2), W, N, G, int(g.integers(0, 1 << 30)), 24, prompt,
                  preseed=bool(case % 3 == 0), variant=variant)


def test_reduction_greedy_and_no_verification():
    cfg = MICRO
    prompt = I.random_prompt(6, cfg.vocab, 3)
    steps, hist = _lossless(cfg, False, 0, 2, 0, 1, 20, prompt)
    assert steps == 20 and hist[1] == 20
    steps, hist = _lossless(cfg, False, 4, 4, 0, 1, 20, prompt)
    assert steps == 20 and hist[1] == 20  # G = 0: no candidates, one token per step
    k = O.Controller(0, 2, 0, 8)
    tok, pos, vis = k.rows(3, 0)
    assert len(tok) == 1 and pos[0] == 0 and vis.tolist() == [[1]]


def test_reduction_prompt_lookup():
    """W = 0 with a prompt-seeded pool: the pool only ever holds prompt
    n-grams, and a prompt that already contains the greedy continuation lets
    whole candidates be accepted."""
    cfg = MICRO
    m = O.Model(cfg, I.make_weights(cfg, 0))
    head = I.random_prompt(5, cfg.vocab, 8)
    cont = O.greedy(m, head, 16)
    prompt = np.concatenate([head, cont, head]).astype(np.int32)
    N, G = 4, 3
    la, steps, hist = O.lookahead(m, prompt, 0, N, G, 16, preseed=True)
    assert np.array_equal(la, O.greedy(m, prompt, 16))
    assert steps < 16
    k = O.Controller(0, N, G, cfg.vocab)
    k.init(prompt, preseed=True)
    grams = {(int(prompt[i]), tuple(int(t) for t in prompt[i + 1:i + N])) for i in range(len(prompt) - N + 1)}
    for key in range(cfg.vocab):
        for v in k.pool(key):
            assert (key, tuple(int(t) for t in v)) in grams
