"""GPU parity of the combined lookahead step against the oracle (through the
C ABI), on the tiny Llama-style workload in fp32 and bf16:

(1) lookahead tokens == the same library's greedy tokens, bit for bit;
(2) rows, emitted tokens, window and pool == the oracle controller fed the
    GPU's argmaxes, bit for bit, every step;
(3) each step's logits within relative L2 error 1e-4 (fp32) / 1e-2 (bf16) of
    the fp32 oracle run on the same weights (single rows: 1e-4 / 2e-2).
"""
import numpy as np
import pytest

import la_inputs as I
import oracle as O
from helpers import build_lib, gpu_decoder, replay_against_oracle

pytestmark = pytest.mark.gpu

TOL = {0: 1e-4, 1: 1e-2}
# (dtype, flags): fp32 SIMT debug path, bf16 on the SIMT kernels, bf16 on the
# tensor-core path (tcgen05 GEMMs), and that path with the step's attention on
# tcgen05 too (LA_ATTN_TC)
MODES = {"fp32": (0, 0), "bf16simt": (1, 8), "bf16": (1, 0), "bf16attntc": (1, 32)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()


def _weights(cfg, bf16):
    return I.make_weights(cfg, 0, bf16=bf16)


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("flags", [0, 4], ids=["graph", "nograph"])
def test_tiny_replay_against_oracle(mode, flags):
    import lossless_lookahead_decoding_gb300 as LA
    dtype, mflags = MODES[mode]
    cfg = I.MODELS["tiny"]
    w = _weights(cfg, dtype == 1)
    W, N, G = I.LOOKAHEAD["tiny"]
    prompt = I.make_prompt("tiny")
    dec = gpu_decoder(cfg, w, dtype, W, N, G, 256, flags=flags | mflags | LA.LA_DEBUG_LOGITS)
    om = O.Model(cfg, w)
    toks, worst = replay_against_oracle(dec, om, prompt, 24, TOL[dtype], row_tol=2 * TOL[dtype] if dtype else None)
    st = dec.stats()
    assert st["steps"] == 24 and st["emitted"] == len(toks)
    dec.close()


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("WNG", [(4, 3, 4), (2, 4, 3), (5, 2, 5), (0, 3, 3), (3, 3, 0)])
def test_lookahead_equals_gpu_greedy(mode, WNG):
    dtype, mflags = MODES[mode]
    cfg = I.MODELS["tiny"]
    w = _weights(cfg, dtype == 1)
    prompt = I.make_prompt("tiny")
    greedy = gpu_decoder(cfg, w, dtype, 0, 2, 0, 256, flags=mflags)
    g = greedy.generate(prompt, 64)
    la = gpu_decoder(cfg, w, dtype, *WNG, 256, flags=mflags)
    t = la.generate(prompt, 64)
    assert np.array_equal(t, g)
    assert greedy.stats()["steps"] == 64
    if WNG[0] > 0 and WNG[2] > 0:
        assert la.stats()["steps"] < 64  # window n-grams got accepted
    if dtype == 0:
        # fp32: also equal to the oracle's greedy output
        assert np.array_equal(g, O.greedy(O.Model(cfg, w), prompt, 64))


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
@pytest.mark.parametrize("WNG", [(64, 2, 63), (42, 4, 0), (31, 3, 32)], ids=["T128", "T127-window", "T127"])
def test_full_and_near_full_steps_equal_greedy(mode, WNG):
    """Steps of 128 and 127 rows (the pass's limit): a 64-column window with
    63 single-token candidates, a 42 x 3 window without verification, and 31
    columns with 32 candidates; lossless against the same library's greedy
    decode, and against the oracle's greedy output in fp32."""
    dtype, mflags = MODES[mode]
    cfg = I.MODELS["tiny"]
    w = _weights(cfg, dtype == 1)
    prompt = I.make_prompt("tiny")
    g = gpu_decoder(cfg, w, dtype, 0, 2, 0, 320, flags=mflags).generate(prompt, 48)
    t = gpu_decoder(cfg, w, dtype, *WNG, 320, flags=mflags).generate(prompt, 48)
    assert np.array_equal(t, g)
    if dtype == 0:
        assert np.array_equal(g, O.greedy(O.Model(cfg, w), prompt, 48))


def test_tiny_fp32_greedy_logits():
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["tiny"]
    w = _weights(cfg, False)
    prompt = I.make_prompt("tiny")
    dec = gpu_decoder(cfg, w, 0, 0, 2, 0, 256, flags=LA.LA_DEBUG_LOGITS)
    ref_t, ref_l = O.greedy(O.Model(cfg, w), prompt, 16, logits=True)
    dec.prefill(prompt)
    for s in range(16):
        e = dec.step()
        assert e[0] == ref_t[s]
        lg = dec.logits()[0]
        assert np.linalg.norm(lg - ref_l[s]) / np.linalg.norm(ref_l[s]) < 1e-4


@pytest.mark.parametrize("mode", ["bf16simt", "bf16", "bf16attntc"])
def test_preseed_and_edge_prompts(mode):
    dtype, mflags = MODES[mode]
    cfg = I.MODELS["tiny"]
    w = _weights(cfg, True)
    greedy = gpu_decoder(cfg, w, 1, 0, 2, 0, 256, flags=mflags)
    la = gpu_decoder(cfg, w, 1, 4, 3, 4, 256, flags=1 | mflags)
    for prompt in (np.array([5], np.int32), np.array([7, 7, 7, 7, 7, 7, 7, 7, 7], np.int32),
                   I.random_prompt(150, cfg.vocab, 3), I.make_prompt("tiny")):
        assert np.array_equal(la.generate(prompt, 40), greedy.generate(prompt, 40))


def test_errors_and_capacity():
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["tiny"]
    w = _weights(cfg, True)
    dec = gpu_decoder(cfg, w, 1, 4, 3, 4, 48, flags=LA.LA_SIMT)
    with pytest.raises(LA.LAError) as e:
        dec.step()
    assert e.value.code == LA.LA_ERR_STATE
    with pytest.raises(LA.LAError) as e:
        dec.prefill(np.arange(50, dtype=np.int32))
    assert e.value.code == LA.LA_ERR_CAPACITY
    with pytest.raises(LA.LAError) as e:
        dec.prefill(np.array([cfg.vocab], np.int32))
    assert e.value.code == LA.LA_ERR_ARG
    dec.prefill(I.make_prompt("tiny"))
    n = 0
    with pytest.raises(LA.LAError) as e:
        for _ in range(100):
            n += len(dec.step())
    assert e.value.code == LA.LA_ERR_CAPACITY
    assert dec.stats()["P"] + 4 + 3 > 48
    with pytest.raises(LA.LAError):
        gpu_decoder(cfg, w, 1, 40, 5, 40, 256)  # 1 + 80*4 rows > 128
    # the tensor-core attention's limits: W + N - 2 <= 31, max_seq <= 4096
    gpu_decoder(cfg, w, 1, 30, 3, 30, 256, flags=LA.LA_ATTN_TC).close()
    gpu_decoder(cfg, w, 1, 31, 3, 31, 256).close()
    for wng, ms in (((31, 3, 31), 256), ((32, 2, 0), 256), ((4, 3, 4), 4096 + 64)):
        with pytest.raises(LA.LAError) as e:
            gpu_decoder(cfg, w, 1, *wng, ms, flags=LA.LA_ATTN_TC)
        assert e.value.code == LA.LA_ERR_ARG


def test_profiled_launches_keep_the_output():
    """The benchmark's profiled pass (LA_PROFILE | LA_NO_GRAPH: CUDA events
    around every kernel class) emits the same tokens as the graph-launched
    greedy decode and reports the tensor-core path's kernel classes."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["tiny"]
    w = _weights(cfg, True)
    W, N, G = I.LOOKAHEAD["tiny"]
    prompt = I.make_prompt("tiny")
    g = gpu_decoder(cfg, w, 1, 0, 2, 0, 256).generate(prompt, 32)
    dec = gpu_decoder(cfg, w, 1, W, N, G, 256, flags=LA.LA_PROFILE | LA.LA_NO_GRAPH)
    assert np.array_equal(dec.generate(prompt, 32), g)
    prof = dec.profile()
    for name in ("gemm_qkv", "gemm_o", "gemm_gateup", "gemm_down", "gemm_lmhead", "attention", "control"):
        assert name in prof and prof[name]["launches"] > 0 and prof[name]["total_ms"] > 0, name
    assert prof["gemm_qkv"]["bytes"] > 0
    dec.close()


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
@pytest.mark.parametrize("WNG", [(4, 3, 4), (5, 4, 3), (3, 2, 3), (2, 5, 2)])
def test_diagonal_levels_against_oracle(mode, WNG):
    """LA_MASK_DIAG: rows, positions, window, pool and emitted tokens
    bit-exact against the oracle controller's diagonal-levels variant fed
    the GPU's argmaxes, logits within the bounds, and the output equal to
    greedy (W < N - 1 included: no n-gram fits a diagonal)."""
    import lossless_lookahead_decoding_gb300 as LA
    dtype, mflags = MODES[mode]
    cfg = I.MODELS["tiny"]
    w = _weights(cfg, dtype == 1)
    prompt = I.make_prompt("tiny")
    dec = gpu_decoder(cfg, w, dtype, *WNG, 256, flags=mflags | LA.LA_MASK_DIAG | LA.LA_DEBUG_LOGITS)
    replay_against_oracle(dec, O.Model(cfg, w), prompt, 16, TOL[dtype], row_tol=2 * TOL[dtype] if dtype else None)
    dec.close()
    g = gpu_decoder(cfg, w, dtype, 0, 2, 0, 256, flags=mflags).generate(prompt, 64)
    la = gpu_decoder(cfg, w, dtype, *WNG, 256, flags=mflags | LA.LA_MASK_DIAG).generate(prompt, 64)
    assert np.array_equal(la, g)


def _override_replay(cfg, w, W, N, G, n_steps, seed, flags=0, max_seq=256, prompt=None):
    """Drive the GPU controller with chosen argmaxes (la_debug_set_argmax_override)
    through every acceptance length, and the oracle controller with the same
    ones: rows, emitted tokens, committed length, window and pool bit-exact
    every step."""
    import lossless_lookahead_decoding_gb300 as LA
    prompt = I.make_prompt("tiny") if prompt is None else prompt
    dec = gpu_decoder(cfg, w, 1, W, N, G, max_seq, flags=flags)
    ctrl = O.Controller(W, N, G, cfg.vocab, variant=O.DIAGONAL if flags & LA.LA_MASK_DIAG else 0)
    ctrl.init(prompt, seed=2, preseed=bool(flags & LA.LA_PRESEED_PROMPT))
    dec.prefill(prompt)
    g = np.random.default_rng(seed)
    vocab = np.unique(prompt)
    c, P = int(prompt[-1]), len(prompt) - 1
    seen = set()
    for step in range(n_steps):
        tok, pos, _ = ctrl.rows(c, P)
        T = len(tok)
        # argmaxes from the prompt's few distinct tokens, so that the pool
        # soon holds n-grams for the current token
        amax = g.choice(vocab, dec.T).astype(np.int32)
        ncand = (T - 1 - W * (N - 1)) // (N - 1)
        if ncand and step % 4:
            # accept the first m tokens of candidate gs: row 0's argmax is its
            # first token, row (gs, i-1)'s its i-th
            gs, m = int(g.integers(0, ncand)), int(g.integers(0, N))
            base = 1 + W * (N - 1) + gs * (N - 1)
            for i in range(m):
                amax[0 if i == 0 else base + i - 1] = tok[base + i]
        dec.override_argmax(amax)
        emit = dec.step()
        tok_g, pos_g, _ = dec.rows()
        assert np.array_equal(tok_g[:T], tok) and np.array_equal(pos_g[:T], pos)
        emit_o, _, _ = ctrl.advance(amax[:T])
        assert np.array_equal(emit, emit_o), (step, emit, emit_o)
        seen.add(len(emit))
        assert np.array_equal(dec.window(), ctrl.window())
        for key in set(int(x) for x in tok):
            assert np.array_equal(dec.pool(key), ctrl.pool(key)), key
        P += len(emit)
        c = int(emit[-1])
    dec.override_argmax(None)
    dec.close()
    return seen


@pytest.mark.parametrize("WNG,flags", [((4, 3, 4), 0), ((5, 4, 3), 0), ((3, 5, 4), 1), ((4, 4, 4), 64)],
                         ids=["columns", "N4", "preseed", "diagonal"])
def test_argmax_override_drives_every_acceptance_length(WNG, flags):
    cfg = I.MODELS["tiny"]
    w = _weights(cfg, True)
    seen = _override_replay(cfg, w, *WNG, 40, seed=sum(WNG) + flags, flags=flags)
    assert seen == set(range(1, WNG[1] + 1)), seen  # 1..N tokens per step all occurred


@pytest.mark.parametrize("mode", ["bf16", "bf16attntc"])
def test_row0_logits_equal_greedy_across_the_merge_paths(mode):
    """Row 0 of every lookahead step (the current token at P) has, bit for
    bit, the logits the greedy decoder computes at P: here at P = 1049..1120,
    where the tcgen05 attention's merge takes its long-context path (rows
    with more than 8 region-A splits of 128 positions, position >= 1071) for
    CTAs that also hold rows of 8 splits, while greedy decoding of those
    rows takes the short path; and the default attention across its
    256-position split boundary at 1024."""
    import lossless_lookahead_decoding_gb300 as LA
    dtype, mflags = MODES[mode]
    cfg = I.MODELS["tiny"]
    w = _weights(cfg, True)
    prompt = I.random_prompt(1050, cfg.vocab, 77)
    la = gpu_decoder(cfg, w, dtype, 15, 5, 15, 1300, flags=mflags | LA.LA_DEBUG_LOGITS)
    g = gpu_decoder(cfg, w, dtype, 0, 2, 0, 1300, flags=mflags | LA.LA_DEBUG_LOGITS)
    la.prefill(prompt)
    g.prefill(prompt)
    P, row0, toks = len(prompt) - 1, {}, []
    while P < 1120:
        emit = la.step()
        row0[P] = la.logits()[0].copy()
        toks.extend(emit.tolist())
        P += len(emit)
    Pg, gt, checked = len(prompt) - 1, [], 0
    while Pg < P:
        e = g.step()
        if Pg in row0:
            assert np.array_equal(g.logits()[0].view(np.uint32), row0[Pg].view(np.uint32)), Pg
            checked += 1
        gt.extend(e.tolist())
        Pg += 1
    assert gt[: len(toks)] == toks[: len(gt)]
    assert checked >= 20 and any(1053 <= p <= 1070 for p in row0)
