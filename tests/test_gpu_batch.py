"""GPU parity of batched decoding (la_create_batch, la_prefill_seq,
la_step_batch): B sequences with prompts of different lengths share each
step's forward pass.  Every sequence's emitted tokens, step rows, argmaxes,
logits, window and pool entries equal, bit for bit, those of a batch-1
context decoding that sequence alone (no row's arithmetic depends on the
other rows of the pass); the batch-1 path is itself pinned to the oracle by
the decode tests, and in fp32 the batched tokens are also compared with the
oracle's greedy output directly.
"""
import numpy as np
import pytest

import la_inputs as I
import oracle as O
from helpers import build_lib

pytestmark = pytest.mark.gpu

# (dtype, flags): fp32 SIMT, bf16 on the SIMT kernels, bf16 tensor-core path
MODES = {"fp32": (0, 0), "bf16simt": (1, 8), "bf16": (1, 0)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()


def _prompts(workload, B, cut=5):
    """B prompts of the workload's recipe with different seeds and lengths."""
    out = []
    for b in range(B):
        p = I.make_prompt(workload, seed=1 + b)
        out.append(p[: len(p) - cut * b])
    return out


def _pair(cfg, w, dtype, WNG, B, flags, max_seq, seed=2):
    """A batched context of B sequences and B batch-1 contexts, same weights."""
    import lossless_lookahead_decoding_gb300 as LA
    dw = LA.device_weights(cfg, w, dtype)
    batched = LA.Decoder(cfg, dw, dtype, *WNG, max_seq, seed=seed, flags=flags, batch=B)
    singles = [LA.Decoder(cfg, dw, dtype, *WNG, max_seq, seed=seed, flags=flags) for _ in range(B)]
    return batched, singles


def _same_state(batched, singles, logits):
    """Debug views of every sequence of the batch == its batch-1 context."""
    for b, s in enumerate(singles):
        batched.select(b)
        tb, pb, nb = batched.rows()
        ts, ps, ns = s.rows()
        assert nb == ns and np.array_equal(tb, ts) and np.array_equal(pb, ps), b
        assert np.array_equal(batched.argmax(), s.argmax()), b
        assert np.array_equal(batched.window(), s.window()), b
        if logits:
            lb, ls = batched.logits(), s.logits()
            assert np.array_equal(lb.view(np.uint32), ls.view(np.uint32)), b
        for key in set(int(x) for x in ts):
            assert np.array_equal(batched.pool(key), s.pool(key)), (b, key)


def _run(batched, singles, prompts, steps, logits=True):
    for b, p in enumerate(prompts):
        batched.prefill_seq(b, p)
        singles[b].prefill(p)
    outs = [[] for _ in prompts]
    for _ in range(steps):
        got = batched.step_batch()
        for b, s in enumerate(singles):
            want = s.step()
            assert np.array_equal(got[b], want), (b, got[b], want)
            outs[b].extend(want.tolist())
        _same_state(batched, singles, logits)
    return outs


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("WNG,B", [((4, 3, 4), 3), ((0, 2, 0), 8), ((5, 4, 3), 4), ((0, 3, 3), 4), ((3, 3, 0), 2),
                                   ((4, 3, 4), 7), ((3, 3, 3), 3), ((0, 2, 0), 40)],
                         ids=["la-b3", "greedy-b8", "la-b4", "promptlookup-b4", "noverify-b2", "la-b7-full",
                              "la-b3-13rows", "greedy-b40"])
def test_batch_equals_batch1_contexts(mode, WNG, B):
    import lossless_lookahead_decoding_gb300 as LA
    dtype, mflags = MODES[mode]
    cfg = I.MODELS["tiny"]
    w = I.make_weights(cfg, 0, bf16=dtype == 1)
    flags = mflags | LA.LA_DEBUG_LOGITS | LA.LA_PRESEED_PROMPT
    batched, singles = _pair(cfg, w, dtype, WNG, B, flags, 256)
    outs = _run(batched, singles, _prompts("tiny", B, cut=3 if B <= 8 else 0), 12)
    st = batched.stats()
    assert st["steps"] == 12 and st["emitted"] == sum(len(o) for o in outs)
    assert st["rows"] == B * (1 + (WNG[0] + WNG[2]) * (WNG[1] - 1))


@pytest.mark.parametrize("flags", [4, 64], ids=["nograph", "diagonal"])
def test_batch_launch_modes_and_mask_variant(flags):
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["tiny"]
    w = I.make_weights(cfg, 0, bf16=True)
    batched, singles = _pair(cfg, w, 1, (4, 3, 4), 3, flags | LA.LA_DEBUG_LOGITS, 256)
    _run(batched, singles, _prompts("tiny", 3, cut=3), 10)


def test_batch_fp32_equals_oracle_greedy():
    """fp32: each sequence of a batch emits the oracle's greedy tokens."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["tiny"]
    w = I.make_weights(cfg, 0)
    B, n = 3, 40
    dw = LA.device_weights(cfg, w, LA.LA_FP32)
    dec = LA.Decoder(cfg, dw, LA.LA_FP32, 4, 3, 4, 256, batch=B)
    prompts = _prompts("tiny", B, cut=4)
    for b, p in enumerate(prompts):
        dec.prefill_seq(b, p)
    outs = [[] for _ in range(B)]
    while min(len(o) for o in outs) < n:
        for b, t in enumerate(dec.step_batch()):
            outs[b].extend(t.tolist())
    om = O.Model(cfg, w)
    for b, p in enumerate(prompts):
        assert np.array_equal(np.array(outs[b][:n], np.int32), O.greedy(om, p, n)), b


@pytest.mark.parametrize("top_k,top_p", [(0, 1.0), (20, 0.7)], ids=["plain", "top20-p0.7"])
def test_batch_sampling_streams(top_k, top_p):
    """Sampling verification: sequence b of a batch draws what a batch-1
    context seeded with seed + b draws (with and without top-k / top-p)."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["tiny"]
    w = I.make_weights(cfg, 0, bf16=True)
    B = 3
    batched, singles = _pair(cfg, w, 1, (4, 3, 4), B, LA.LA_DEBUG_LOGITS, 256)
    batched.set_sampling(0.9, 11, top_k=top_k, top_p=top_p)
    for b, s in enumerate(singles):
        s.set_sampling(0.9, 11 + b, top_k=top_k, top_p=top_p)
    _run(batched, singles, _prompts("tiny", B, cut=3), 16)


def test_batch_7b_widths_two_layer_slice():
    """7B widths (tcgen05 GEMMs at d 4096, FFN 11008, vocab 32000; 32 heads
    x 128): two sequences of 57 rows (W=7 N=5 G=7) fill 114 of a pass's 128
    rows; 512- and 496-token prompts."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["7b"].sliced(2)
    full = I.make_weights(I.MODELS["7b"], 0, bf16=True, layers=[0, 1])
    w = {k: (v[:2] if isinstance(v, list) else v) for k, v in full.items()}
    batched, singles = _pair(cfg, w, 1, (7, 5, 7), 2, LA.LA_DEBUG_LOGITS, 640)
    _run(batched, singles, _prompts("7b", 2, cut=16), 4)


@pytest.mark.parametrize("WNG,B", [((0, 2, 0), 8), ((0, 2, 0), 3), ((3, 3, 3), 2)],
                         ids=["greedy-b8", "greedy-b3", "la-13rows-b2"])
def test_batch_narrow_attention_7b_widths(WNG, B):
    """Batches of at most 16 rows per sequence run the attention's narrow
    instances (at most 8 rows and more CTAs than SMs: 2 warps, three CTAs
    per SM; otherwise 4 warps, two per SM) at head_dim 128: 470-512-token
    prompts (two 256-position splits and a tail), every sequence against its
    batch-1 context (wide instance), bit for bit."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["7b"].sliced(2)
    full = I.make_weights(I.MODELS["7b"], 0, bf16=True, layers=[0, 1])
    w = {k: (v[:2] if isinstance(v, list) else v) for k, v in full.items()}
    batched, singles = _pair(cfg, w, 1, WNG, B, LA.LA_DEBUG_LOGITS, 640)
    _run(batched, singles, _prompts("7b", B, cut=16), 3)


@pytest.mark.parametrize("B", [3, 24])
def test_batch_narrow_attention_34b_gqa_greedy(B):
    """Greedy batches at 34B widths: the narrow instances stack the 8 query
    heads of a KV head as rows of the 16-row tile (3 sequences: 24 CTAs a
    split, the 4-warp instance; 24 sequences: 192, the 2-warp one); the
    first, a middle and the last sequence against batch-1 contexts, bit for
    bit."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["34b"].sliced(1)
    full = I.make_weights(I.MODELS["34b"], 0, bf16=True, layers=[0])
    w = {k: (v[:1] if isinstance(v, list) else v) for k, v in full.items()}
    dw = LA.device_weights(cfg, w, LA.LA_BF16)
    flags = LA.LA_DEBUG_LOGITS
    prompts = [I.plant_spans(I.zipf_tokens(300 - 7 * b, 4000, 1.2, 21 + b), 16, 6, 22 + b) for b in range(B)]
    batched = LA.Decoder(cfg, dw, LA.LA_BF16, 0, 2, 0, 384, flags=flags, batch=B)
    for b, p in enumerate(prompts):
        batched.prefill_seq(b, p)
    picks = sorted({0, B // 2, B - 1})
    singles = {b: LA.Decoder(cfg, dw, LA.LA_BF16, 0, 2, 0, 384, flags=flags) for b in picks}
    for b, d in singles.items():
        d.prefill(prompts[b])
    for _ in range(3):
        got = batched.step_batch()
        for b, d in singles.items():
            assert np.array_equal(got[b], d.step()), b
            batched.select(b)
            assert np.array_equal(batched.logits().view(np.uint32), d.logits().view(np.uint32)), b
    for d in [batched] + list(singles.values()):
        d.close()


def test_batch_34b_widths_gqa_one_layer_slice():
    """34B widths with grouped-query attention (64 query heads on 8 KV heads,
    d 8192): two sequences at the 34B setting W=7 N=5 G=7."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["34b"].sliced(1)
    full = I.make_weights(I.MODELS["34b"], 0, bf16=True, layers=[0])
    w = {k: (v[:1] if isinstance(v, list) else v) for k, v in full.items()}
    prompts = [I.plant_spans(I.zipf_tokens(256 - 24 * b, 4000, 1.2, 11 + b), 16, 6, 12 + b) for b in range(2)]
    batched, singles = _pair(cfg, w, 1, (7, 5, 7), 2, LA.LA_DEBUG_LOGITS | LA.LA_PRESEED_PROMPT, 384)
    _run(batched, singles, prompts, 4)


def test_batch_errors():
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["tiny"]
    w = I.make_weights(cfg, 0, bf16=True)
    dw = LA.device_weights(cfg, w, LA.LA_BF16)
    with pytest.raises(LA.LAError):  # 8 x 17 rows > 128
        LA.Decoder(cfg, dw, LA.LA_BF16, 4, 3, 4, 256, batch=8)
    with pytest.raises(LA.LAError):  # the tcgen05 attention serves one sequence
        LA.Decoder(cfg, dw, LA.LA_BF16, 4, 3, 4, 256, flags=LA.LA_ATTN_TC, batch=2)
    dec = LA.Decoder(cfg, dw, LA.LA_BF16, 4, 3, 4, 256, batch=2)
    p = I.make_prompt("tiny")
    with pytest.raises(LA.LAError) as e:
        dec.prefill(p)
    assert e.value.code == LA.LA_ERR_STATE
    with pytest.raises(LA.LAError) as e:
        dec.prefill_seq(2, p)
    assert e.value.code == LA.LA_ERR_ARG
    dec.prefill_seq(0, p)
    with pytest.raises(LA.LAError) as e:  # sequence 1 not prefilled yet
        dec.step_batch()
    assert e.value.code == LA.LA_ERR_STATE
    dec.prefill_seq(1, p[:20])
    with pytest.raises(LA.LAError) as e:
        dec.step()
    assert e.value.code == LA.LA_ERR_STATE
    with pytest.raises(LA.LAError) as e:
        dec.select(5)
    assert e.value.code == LA.LA_ERR_ARG
    a, b = dec.step_batch()
    assert 1 <= len(a) <= 3 and 1 <= len(b) <= 3
    # a full cache in one sequence stops the batch
    small = LA.Decoder(cfg, dw, LA.LA_BF16, 4, 3, 4, 48, batch=2)
    small.prefill_seq(0, p[:8])
    small.prefill_seq(1, p[:40])
    with pytest.raises(LA.LAError) as e:
        for _ in range(16):
            small.step_batch()
    assert e.value.code == LA.LA_ERR_CAPACITY


def test_batch_7b_full_depth():
    """The full 32-layer 7B model: two sequences (W=7 N=5 G=7, 512- and
    496-token prompts) in one pass equal their batch-1 decodings bit for bit
    (tokens, rows, argmaxes, windows, pools) for 8 steps, and sequence 0's
    tokens equal the same library's greedy decode of its prompt."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["7b"]
    dw = LA.device_weights(cfg, I.iter_weights(cfg, 0, bf16=False), LA.LA_BF16)
    batched = LA.Decoder(cfg, dw, LA.LA_BF16, 7, 5, 7, 640, batch=2)
    singles = [LA.Decoder(cfg, dw, LA.LA_BF16, 7, 5, 7, 640) for _ in range(2)]
    prompts = _prompts("7b", 2, cut=16)
    outs = _run(batched, singles, prompts, 8, logits=False)
    for d in [batched] + singles:
        d.close()
    greedy = LA.Decoder(cfg, dw, LA.LA_BF16, 0, 2, 0, 640)
    g = greedy.generate(prompts[0], len(outs[0]))
    greedy.close()
    assert np.array_equal(np.array(outs[0], np.int32), g)


@pytest.mark.parametrize("WNG,B", [((0, 2, 0), 128), ((1, 2, 0), 64)], ids=["greedy-b128", "w1-b64"])
def test_batch_fills_the_128_row_pass(WNG, B):
    """A pass of exactly 128 rows on the tcgen05 GEMMs at 7B widths (2-layer
    slice): 128 greedy sequences, or 64 of two rows; the first, a middle and
    the last sequence against their batch-1 contexts, bit for bit."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["7b"].sliced(2)
    full = I.make_weights(I.MODELS["7b"], 0, bf16=True, layers=[0, 1])
    w = {k: (v[:2] if isinstance(v, list) else v) for k, v in full.items()}
    dw = LA.device_weights(cfg, w, LA.LA_BF16)
    flags = LA.LA_DEBUG_LOGITS
    batched = LA.Decoder(cfg, dw, LA.LA_BF16, *WNG, 320, flags=flags, batch=B)
    prompts = [I.random_prompt(64 + (7 * b) % 97, cfg.vocab, 100 + b) for b in range(B)]
    for b, p in enumerate(prompts):
        batched.prefill_seq(b, p)
    picks = [0, B // 2, B - 1]
    singles = {b: LA.Decoder(cfg, dw, LA.LA_BF16, *WNG, 320, flags=flags) for b in picks}
    for b, d in singles.items():
        d.prefill(prompts[b])
    for _ in range(3):
        got = batched.step_batch()
        assert all(1 <= len(t) <= WNG[1] for t in got)
        for b, d in singles.items():
            assert np.array_equal(got[b], d.step()), b
            batched.select(b)
            assert np.array_equal(batched.argmax(), d.argmax()), b
            assert np.array_equal(batched.logits().view(np.uint32), d.logits().view(np.uint32)), b
    for d in [batched] + list(singles.values()):
        d.close()


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_generate_batch_equals_batch1_generate(mode):
    """la_generate_batch: every sequence's max_new tokens equal la_generate of
    a batch-1 context on its prompt (bit for bit); a cache that fills first
    returns LA_ERR_CAPACITY."""
    import lossless_lookahead_decoding_gb300 as LA
    dtype, mflags = MODES[mode]
    cfg = I.MODELS["tiny"]
    w = I.make_weights(cfg, 0, bf16=dtype == 1)
    dw = LA.device_weights(cfg, w, dtype)
    prompts = _prompts("tiny", 3, cut=7)
    dec = LA.Decoder(cfg, dw, dtype, 4, 3, 4, 256, flags=mflags, batch=3)
    got = dec.generate_batch(prompts, 40)
    one = LA.Decoder(cfg, dw, dtype, 4, 3, 4, 256, flags=mflags)
    for b, p in enumerate(prompts):
        assert len(got[b]) == 40
        assert np.array_equal(got[b], one.generate(p, 40)), b
    assert dec.stats()["emitted"] >= 3 * 40
    small = LA.Decoder(cfg, dw, dtype, 4, 3, 4, 64, flags=mflags, batch=3)
    with pytest.raises(LA.LAError) as e:
        small.generate_batch(prompts, 60)
    assert e.value.code == LA.LA_ERR_CAPACITY
