"""Pins of the oracle's sampling verification (R10) and temperature sampling.

The summary page says lookahead decoding supports sampling and keeps the
output distribution exactly; it gives no algorithm, so the rule is designed
here (see the oracle's header).  What fixes it, independently of the oracle:

* the rule's output distribution, evaluated exactly in rational arithmetic
  over every accept/reject branch, equals the target softmax;
* the oracle's sampler agrees with the softmax it samples from (Monte Carlo);
* on a Markov toy model (a row's next-token logits depend only on the row's
  own token), the token sequences of the sampled lookahead process agree with
  the exact probabilities of plain ancestral sampling (Monte Carlo);
* structural facts of one verification step: a candidate value is emitted
  only by being accepted, and then the step continues to the next level;
* tau -> 0 reduces sampled decoding and sampled lookahead to greedy decoding;
* top-k (another sampling scheme the summary page says is supported): draws
  stay inside the top-k tokens by weight (computed here from the per-token
  weights, ties to the lower index), follow the softmax renormalised over
  them, and the sampled lookahead with top-k matches top-k ancestral sampling
  on the Markov model; top_k >= V is plain sampling, top_k = 1 deterministic;
* top-p (nucleus sampling, Holtzman et al. 2020): on a distribution printed
  here (0.5, 0.3, 0.15, 0.05) the kept sets for p = 0.45, 0.75, 0.9 are {0},
  {0, 1}, {0, 1, 2}, and draws follow the renormalised probabilities; after
  top_k = 2 the bound applies to the renormalised pair (0.625, 0.375); equal
  weights are kept lower index first; top_p = 1 is plain sampling and a tiny
  top_p is greedy; the sampled lookahead with top-p matches top-p ancestral
  sampling on the Markov model;
* the fp32 exponential the probabilities are built from is within 3 ulp of
  the library exponential over its whole range (2 ulp; measured 1.24), exact at 0 and at integer
  multiples of ln 2 where the polynomial sees t = 0, and flushes to 0 below
  2^-125.
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np
import pytest

import la_inputs as I
import oracle as O


def _level_rule_exact(p, cands):
    """Exact output distribution of one verification level: distinct
    candidate values tried in order, v accepted with probability
    p(v) / (1 - rejected mass), else the token drawn from p without the
    rejected values."""
    out = [Fraction(0)] * len(p)
    reach, rej_mass, rejected = Fraction(1), Fraction(0), []
    for v in cands:
        if v in rejected:
            continue
        left = 1 - rej_mass
        a = p[v] / left if left > 0 else Fraction(1)
        out[v] += reach * a
        reach *= 1 - a
        rejected.append(v)
        rej_mass += p[v]
    left = 1 - rej_mass
    for v in range(len(p)):
        if v not in rejected and left > 0:
            out[v] += reach * p[v] / left
    return out


def test_verification_rule_is_exact_in_rationals():
    rng = np.random.default_rng(0)
    for _ in range(300):
        V = int(rng.integers(2, 7))
        w = [int(x) for x in rng.integers(0, 6, V)]
        if sum(w) == 0:
            w[0] = 1
        p = [Fraction(x, sum(w)) for x in w]
        k = int(rng.integers(0, 6))
        cands = [int(x) for x in rng.integers(0, V, k)]  # duplicates and zero-mass values included
        assert _level_rule_exact(p, cands) == p, (p, cands)


def _softmax(z, tau):
    z = np.asarray(z, np.float64) / tau
    e = np.exp(z - z.max())
    return e / e.sum()


def _close(freq, p, n, k=5.0):
    return np.all(np.abs(freq - p) <= k * np.sqrt(p * (1 - p) / n) + 2e-4)


@pytest.mark.parametrize("tau", [0.7, 2.0])
def test_sampler_matches_softmax(tau):
    z = np.random.default_rng(1).normal(0, 1.5, 8).astype(np.float32)
    n = 200_000
    x = O.sample_logits(z, tau, O.Rng(11), n)
    freq = np.bincount(x, minlength=8) / n
    assert _close(freq, _softmax(z, tau), n), (freq, _softmax(z, tau))


def test_one_step_structure_and_level_distributions():
    """W = 0, N = 2: row 0 and one row per candidate.  The first token follows
    row 0's softmax; a candidate value is emitted only when accepted, and then
    the bonus token follows the softmax of that candidate's row."""
    V, c, tau = 8, 2, 1.0
    rng = np.random.default_rng(2)
    ctrl = O.Controller(0, 2, 4, V)
    ctrl.init(np.array([c], np.int32))
    for v in (3, 1, 3, 5):  # the duplicate value is dropped by the pool
        ctrl.insert(c, [v])
    tok, pos, vis = ctrl.rows(c, 10)
    T = len(tok)
    assert list(tok) == [c, 3, 1, 5]
    logits = rng.normal(0, 1.2, (T, V)).astype(np.float32)
    r = O.Rng(3)
    n = 120_000
    first = np.zeros(V)
    second = {v: np.zeros(V) for v in (3, 1, 5)}
    for _ in range(n):
        ctrl.rows(c, 10)
        emit, rows, g = ctrl.advance_sample(logits, tau, r)
        first[emit[0]] += 1
        if emit[0] in (3, 1, 5):
            assert len(emit) == 2 and list(rows) == [0, 1 + [3, 1, 5].index(emit[0])]
            second[emit[0]][emit[1]] += 1
        else:
            assert len(emit) == 1 and g == -1
    assert _close(first / n, _softmax(logits[0], tau), n)
    for i, v in enumerate((3, 1, 5)):
        m = second[v].sum()
        assert m > 200
        assert _close(second[v] / m, _softmax(logits[1 + i], tau), m)


@pytest.mark.parametrize("W,N,G", [(2, 3, 3), (0, 4, 2)])
def test_sampled_lookahead_matches_ancestral_sampling_on_markov_model(W, N, G):
    """Token sequences of length K from the sampled lookahead process (window,
    pool, harvest and all) against the exact probabilities of sampling the
    Markov chain token by token."""
    V, K, tau = 5, 3, 1.0
    Z = (np.random.default_rng(4).normal(0, 1.6, (V, V))).astype(np.float32)
    P1 = np.stack([_softmax(Z[a], tau) for a in range(V)])
    prompt = np.array([0, 1, 2, 1, 0, 3, 1, 2, 4, 1], np.int32)
    c0 = int(prompt[-1])
    ctrl = O.Controller(W, N, G, V)
    ctrl.init(prompt, seed=5, preseed=True)
    r = O.Rng(6)
    n = 40_000
    counts = np.zeros((V,) * K)
    steps = toks = 0
    for _ in range(n):
        c, P, out = c0, 9, []
        while len(out) < K:
            tok, pos, vis = ctrl.rows(c, P)
            emit, rows, g = ctrl.advance_sample(Z[tok], tau, r)
            out.extend(emit.tolist())
            steps += 1
            toks += len(emit)
            c, P = int(emit[-1]), P + len(emit)
        counts[tuple(out[:K])] += 1
    assert toks / steps > 1.1  # candidates do get accepted
    exact = np.zeros((V,) * K)
    for seq in itertools.product(range(V), repeat=K):
        pr, prev = 1.0, c0
        for t in seq:
            pr *= P1[prev, t]
            prev = t
        exact[seq] = pr
    freq = counts / n
    assert _close(freq.ravel(), exact.ravel(), n)
    m = exact.ravel() > 0
    chi2 = float((((counts.ravel() - n * exact.ravel()) ** 2)[m] / (n * exact.ravel()[m])).sum())
    assert chi2 < (V ** K - 1) + 6 * np.sqrt(2 * (V ** K - 1)), chi2


@pytest.fixture(scope="module")
def tiny():
    cfg = I.MODELS["tiny"]
    w = I.make_weights(cfg, 0, bf16=False)
    return cfg, O.Model(cfg, w), I.make_prompt("tiny")


def test_tau_to_zero_is_greedy(tiny):
    cfg, m, prompt = tiny
    g, lg = O.greedy(m, prompt, 48, logits=True)
    top2 = np.sort(lg, axis=1)[:, -2:]
    assert (top2[:, 1] - top2[:, 0]).min() > 1e-5  # no near-tie for the argmax
    tau = 1e-8
    assert np.array_equal(O.sample_decode(m, prompt, 48, tau, 9), g)
    W, N, G = I.LOOKAHEAD["tiny"]
    t, steps, _ = O.lookahead_sample(m, prompt, W, N, G, 48, tau, 9)
    assert np.array_equal(t, g)
    assert steps < 48


def test_sampled_lookahead_runs_and_is_reproducible(tiny):
    cfg, m, prompt = tiny
    W, N, G = I.LOOKAHEAD["tiny"]
    a = O.lookahead_sample(m, prompt, W, N, G, 40, 0.5, 21)
    b = O.lookahead_sample(m, prompt, W, N, G, 40, 0.5, 21)
    assert np.array_equal(a[0], b[0]) and a[1] == b[1]
    assert a[2].sum() == a[1] and (a[0] >= 0).all() and (a[0] < cfg.vocab).all()
    s1 = O.sample_decode(m, prompt, 40, 0.5, 21)
    s2 = O.sample_decode(m, prompt, 40, 0.5, 21)
    assert np.array_equal(s1, s2)


def test_sampling_exponential_against_the_library():
    xs = np.concatenate([-np.linspace(0.0, 86.6, 200001), -np.geomspace(1e-8, 1.0, 2001)]).astype(np.float32)
    got = np.array([O.exp_neg(float(x)) for x in xs], np.float64)
    ref = np.exp(xs.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() <= 2 * 2.0 ** -24, rel.max()  # measured 1.24 ulp
    assert O.exp_neg(0.0) == 1.0
    # x = -k ln 2 up to float rounding of the argument: 2^-k to a few ulp
    for k in range(0, 126, 5):
        x = np.float32(-k * np.log(2.0))
        assert abs(O.exp_neg(float(x)) / np.exp(np.float64(x)) - 1) <= 3 * 2.0 ** -24
    assert O.exp_neg(-87.0) == 0.0 and O.exp_neg(-1e4) == 0.0
    # monotone over a fine grid
    assert (np.diff(got[:200001]) <= 0).all()


@pytest.mark.parametrize("V", [7, 1000, 32000])
def test_integer_weights_are_the_softmax(V):
    """The weights E(v) = floor(e(v) 2^B), B = 63 - ceil(log2(V + 1)): the
    maximum has weight exactly 2^B, the total stays below 2^63, and E / S is
    the temperature softmax wherever it is above 1e-9, to within the fp32
    roundings of the argument x = (z - max) / tau (two: |x| 2^-23) and a few
    ulp of the exponential -- for the token and for the normaliser."""
    B = 63 - int(np.ceil(np.log2(V + 1)))
    g = np.random.default_rng(V)
    z = (g.standard_normal(V) * 4).astype(np.float32)
    for tau in (0.3, 0.7, 1.5):
        mx = float(z.max())
        E = np.array([O.sample_weight(float(x), mx, tau, V) for x in z], dtype=object)
        assert E[int(z.argmax())] == 2 ** B
        S = int(sum(E))
        assert S < 2 ** 63
        p = np.array([int(e) / S for e in E])
        ref = np.exp((z.astype(np.float64) - mx) / tau)
        ref /= ref.sum()
        big = ref > 1e-9
        x = np.abs((z.astype(np.float64) - mx) / tau)
        tol = 2 * (2 * x[big].max() + 4) * 2.0 ** -24
        assert np.abs(p[big] / ref[big] - 1).max() <= tol


# ------------------------------------------------------------------ top-k

def _top_k_set(z, tau, k):
    """The top-k tokens by the integer weights (ties to the lower index),
    computed here from the per-token weights, apart from the oracle's own
    restriction."""
    V = len(z)
    mx = float(np.max(z))
    E = [O.sample_weight(float(x), mx, tau, V) for x in z]
    order = sorted(range(V), key=lambda v: (-E[v], v))
    return set(order[:k]), E


@pytest.mark.parametrize("k", [1, 2, 5, 7])
def test_top_k_draws_follow_the_restricted_softmax(k):
    """Draws with top_k = k only ever pick the k tokens of largest weight and
    follow the softmax renormalised over them; k = 1 is deterministic."""
    V, tau, n = 8, 0.9, 120_000
    z = np.random.default_rng(7).normal(0, 1.3, V).astype(np.float32)
    keep, E = _top_k_set(z, tau, k)
    x = O.sample_logits(z, tau, O.Rng(13), n, top_k=k)
    assert set(np.unique(x).tolist()) <= keep
    p = np.zeros(V)
    sm = _softmax(z, tau)
    for v in keep:
        p[v] = sm[v]
    p /= p.sum()
    freq = np.bincount(x, minlength=V) / n
    assert _close(freq, p, n), (freq, p)
    if k == 1:
        assert len(np.unique(x)) == 1


def test_top_k_of_the_whole_vocabulary_is_plain_sampling():
    """top_k = 0, = V and > V draw exactly what plain sampling draws from the
    same uniform stream; the key order puts equal weights lower index first."""
    V = 9
    z = np.random.default_rng(8).normal(0, 1.0, V).astype(np.float32)
    ref = O.sample_logits(z, 1.3, O.Rng(21), 500)
    for k in (0, V, V + 5):
        assert np.array_equal(O.sample_logits(z, 1.3, O.Rng(21), 500, top_k=k), ref)
    assert O.top_k_key(7, 2, 10) > O.top_k_key(7, 3, 10) > O.top_k_key(6, 0, 10)


def test_top_k_ties_go_to_the_lower_index():
    """Equal logits give equal weights; top_k keeps the lowest indices among
    them."""
    z = np.array([0.5, 1.0, 1.0, 1.0, -2.0], np.float32)
    x = O.sample_logits(z, 1.0, O.Rng(5), 20_000, top_k=2)
    assert set(np.unique(x).tolist()) == {1, 2}


@pytest.mark.parametrize("W,N,G,k", [(2, 3, 3, 2), (0, 4, 2, 3)])
def test_sampled_lookahead_with_top_k_matches_ancestral_top_k_sampling(W, N, G, k):
    """As the Markov-model test above, with every row restricted to its top_k
    tokens: the lookahead process's token sequences against the exact
    probabilities of top-k ancestral sampling."""
    V, K, tau = 5, 3, 1.0
    Z = (np.random.default_rng(4).normal(0, 1.6, (V, V))).astype(np.float32)
    P1 = np.zeros((V, V))
    for a in range(V):
        keep, _ = _top_k_set(Z[a], tau, k)
        sm = _softmax(Z[a], tau)
        for v in keep:
            P1[a, v] = sm[v]
        P1[a] /= P1[a].sum()
    prompt = np.array([0, 1, 2, 1, 0, 3, 1, 2, 4, 1], np.int32)
    c0 = int(prompt[-1])
    ctrl = O.Controller(W, N, G, V)
    ctrl.init(prompt, seed=5, preseed=True)
    r = O.Rng(9)
    n = 40_000
    counts = np.zeros((V,) * K)
    for _ in range(n):
        c, P, out = c0, 9, []
        while len(out) < K:
            tok, pos, vis = ctrl.rows(c, P)
            emit, rows, g = ctrl.advance_sample(Z[tok], tau, r, top_k=k)
            out.extend(emit.tolist())
            c, P = int(emit[-1]), P + len(emit)
        counts[tuple(out[:K])] += 1
    exact = np.zeros((V,) * K)
    for seq in itertools.product(range(V), repeat=K):
        pr, prev = 1.0, c0
        for t in seq:
            pr *= P1[prev, t]
            prev = t
        exact[seq] = pr
    assert counts.ravel()[exact.ravel() == 0].sum() == 0  # nothing outside the top-k sets
    freq = counts / n
    assert _close(freq.ravel(), exact.ravel(), n)


# ------------------------------------------------------------------ top-p

_P4 = np.array([0.5, 0.3, 0.15, 0.05])


def _draw_freq(z, tau, n, seed, **kw):
    x = O.sample_logits(z, tau, O.Rng(seed), n, **kw)
    return x, np.bincount(x, minlength=len(z)) / n


@pytest.mark.parametrize("top_p,keep", [(0.45, [0]), (0.75, [0, 1]), (0.9, [0, 1, 2]), (0.99, [0, 1, 2, 3])])
def test_top_p_keeps_the_nucleus_of_a_printed_distribution(top_p, keep):
    """p = (0.5, 0.3, 0.15, 0.05) as logits log p at tau = 1: the smallest
    leading set holding top_p of the mass, and draws from it renormalised."""
    z = np.log(_P4).astype(np.float32)
    n = 100_000
    x, freq = _draw_freq(z, 1.0, n, 31, top_p=top_p)
    assert sorted(np.unique(x).tolist()) == keep
    q = np.zeros(4)
    q[keep] = _P4[keep]
    q /= q.sum()
    assert _close(freq, q, n), (freq, q)


@pytest.mark.parametrize("top_p,keep", [(0.6, [0]), (0.7, [0, 1]), (0.99, [0, 1])])
def test_top_p_applies_to_the_top_k_renormalised(top_p, keep):
    """top_k = 2 leaves (0.5, 0.3) renormalised to (0.625, 0.375): top_p 0.6
    keeps token 0 alone, 0.7 both; token 2 never appears."""
    z = np.log(_P4).astype(np.float32)
    x, _ = _draw_freq(z, 1.0, 40_000, 32, top_k=2, top_p=top_p)
    assert sorted(np.unique(x).tolist()) == keep


def test_top_p_ties_go_to_the_lower_index():
    """Equal logits: (1, 1, 1, 0) has weights w, w, w, w/e; half the mass
    (1.68 w) needs two of the equal tokens, the lower two."""
    z = np.array([1.0, 1.0, 1.0, 0.0], np.float32)
    x, _ = _draw_freq(z, 1.0, 20_000, 33, top_p=0.5)
    assert sorted(np.unique(x).tolist()) == [0, 1]


def test_top_p_one_is_plain_sampling_and_tiny_top_p_is_greedy():
    """top_p = 1 draws exactly what plain sampling draws from the same
    stream; top_p -> 0 leaves the argmax alone (greedy decoding)."""
    z = np.random.default_rng(12).normal(0, 1.0, 11).astype(np.float32)
    ref = O.sample_logits(z, 0.8, O.Rng(41), 600)
    assert np.array_equal(O.sample_logits(z, 0.8, O.Rng(41), 600, top_p=1.0), ref)
    x = O.sample_logits(z, 0.8, O.Rng(41), 600, top_p=1e-6)
    assert np.all(x == int(np.argmax(z)))
    assert O.top_p24(1.0) == 1 << 24 and O.top_p24(0.5) == 1 << 23 and O.top_p24(1e-12) == 1
    assert O.top_p24(0.9) == int(np.floor(np.float64(np.float32(0.9)) * 2.0**24))


def test_top_p_mass_boundary_is_inclusive():
    """Weights (w, w): top_p = 0.5 is reached exactly by the first token, so
    only token 0 is kept; just above 0.5 both are."""
    z = np.array([0.0, 0.0], np.float32)
    x, _ = _draw_freq(z, 1.0, 4_000, 34, top_p=0.5)
    assert np.all(x == 0)
    x, _ = _draw_freq(z, 1.0, 4_000, 34, top_p=0.5 + 2.0**-20)
    assert sorted(np.unique(x).tolist()) == [0, 1]


@pytest.mark.parametrize("W,N,G,k,top_p", [(2, 3, 3, 0, 0.8), (0, 4, 2, 4, 0.7)])
def test_sampled_lookahead_with_top_p_matches_ancestral_top_p_sampling(W, N, G, k, top_p):
    """The Markov-model test with every row restricted by top-k (k > 0) and
    then top-p: the lookahead process's token sequences against the exact
    probabilities of that ancestral sampling, the kept sets computed here
    from the probabilities in float64 (no kept set of this model has mass
    within 1e-6 of the bound)."""
    V, K, tau = 5, 3, 1.0
    Z = (np.random.default_rng(4).normal(0, 1.6, (V, V))).astype(np.float32)
    P1 = np.zeros((V, V))
    for a in range(V):
        sm = _softmax(Z[a], tau)
        order = sorted(range(V), key=lambda v: (-sm[v], v))
        if k:
            order = order[:k]
        tot = sum(sm[v] for v in order)
        acc = 0.0
        for v in order:
            assert abs(acc / tot - top_p) > 1e-6
            P1[a, v] = sm[v]
            acc += sm[v]
            if acc / tot >= top_p:
                break
        P1[a] /= P1[a].sum()
    prompt = np.array([0, 1, 2, 1, 0, 3, 1, 2, 4, 1], np.int32)
    c0 = int(prompt[-1])
    ctrl = O.Controller(W, N, G, V)
    ctrl.init(prompt, seed=5, preseed=True)
    r = O.Rng(19)
    n = 40_000
    counts = np.zeros((V,) * K)
    for _ in range(n):
        c, P, out = c0, 9, []
        while len(out) < K:
            tok, pos, vis = ctrl.rows(c, P)
            emit, rows, g = ctrl.advance_sample(Z[tok], tau, r, top_k=k, top_p=top_p)
            out.extend(emit.tolist())
            c, P = int(emit[-1]), P + len(emit)
        counts[tuple(out[:K])] += 1
    exact = np.zeros((V,) * K)
    for seq in itertools.product(range(V), repeat=K):
        pr, prev = 1.0, c0
        for t in seq:
            pr *= P1[prev, t]
            prev = t
        exact[seq] = pr
    assert counts.ravel()[exact.ravel() == 0].sum() == 0  # nothing outside the kept sets
    freq = counts / n
    assert _close(freq.ravel(), exact.ravel(), n)
