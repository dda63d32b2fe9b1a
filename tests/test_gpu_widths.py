"""GPU parity at realistic widths through the C ABI:

* a GQA decoder with head_dim 128 (4 query heads share 1 KV head) and a
  300-token prompt, so the tensor-core attention walks several shared chunks
  and two 256-position splits before its tail chunks;
* a 2-layer slice of the Llama-2-7B-shaped workload (d 4096, 32 heads x 128,
  FFN 11008, vocab 32000, the 512-token planted-span prompt, W=15 N=5 G=15,
  121 rows per step) -- the full widths the benchmark runs, with the oracle
  on the same bytes;
* a 1-layer slice of the Llama-2-13B-shaped workload (d 5120, 40 heads x
  128, FFN 13824, the 1024-token prompt, W=10 N=5 G=10, 81 rows per step);
* a 1-layer slice of the CodeLlama-34B-shaped workload (d 8192, 64 query
  heads sharing 8 KV heads, FFN 22016, vocab 32000, W=7 N=5 G=7 with the
  prompt-seeded pool, 57 rows per step) on a 256-token Zipf(1.2) prompt
  over 4000 ids with planted spans (shorter than the benchmark's 2048 so the
  oracle's prefill stays within seconds).

* the full-depth 7B-, 13B- and 34B-shaped models in the configurations the
  benchmark times (no debug logits): the oracle cannot run those forwards in
  seconds, so there only what holds at any size is checked
  -- every step's rows, emitted tokens, window and pool bit-exact against the
  oracle controller fed the GPU's argmaxes, and the tokens equal to GPU greedy.

Checks: each step's logits within relative L2 error 1e-2 (bf16) of the fp32
oracle's (every row within 2e-2: a CPU emulation of the kernels' bf16 rounding
points gives ~1.1e-2 for single rows of the 2-layer 7B slice), rows/window/pool/emitted tokens bit-exact against the oracle
controller fed the GPU's argmaxes, and lookahead tokens == GPU greedy tokens.
"""
import numpy as np
import pytest

import la_inputs as I
import oracle as O
from helpers import build_lib, gpu_decoder, replay_against_oracle

pytestmark = pytest.mark.gpu

GQA = I.ModelConfig("gqa-hd128", 2, 512, 4, 1, 128, 1024, 2048)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()


@pytest.mark.parametrize("flags", [0, 8, 32], ids=["tc", "simt", "attntc"])
def test_gqa_hd128_long_prompt(flags):
    import lossless_lookahead_decoding_gb300 as LA
    cfg = GQA
    w = I.make_weights(cfg, 0, bf16=True)
    prompt = I.plant_spans(I.zipf_tokens(300, cfg.vocab, 1.1, 7), 16, 4, 8)
    W, N, G = 7, 5, 7
    dec = gpu_decoder(cfg, w, 1, W, N, G, 512, flags=flags | LA.LA_DEBUG_LOGITS)
    toks, worst = replay_against_oracle(dec, O.Model(cfg, w), prompt, 6, 1e-2, row_tol=2e-2)
    g = gpu_decoder(cfg, w, 1, 0, 2, 0, 512, flags=flags).generate(prompt, 48)
    la = gpu_decoder(cfg, w, 1, W, N, G, 512, flags=flags).generate(prompt, 48)
    assert np.array_equal(la, g)


@pytest.mark.parametrize("flags", [0, 32], ids=["tc", "attntc"])
def test_7b_width_two_layer_slice(flags):
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["7b"].sliced(2)
    full = I.make_weights(I.MODELS["7b"], 0, bf16=True, layers=[0, 1])
    w = {k: (v[:2] if isinstance(v, list) else v) for k, v in full.items()}
    prompt = I.make_prompt("7b")
    W, N, G = I.LOOKAHEAD["7b"]
    dec = gpu_decoder(cfg, w, 1, W, N, G, 640, flags=flags | LA.LA_DEBUG_LOGITS)
    toks, worst = replay_against_oracle(dec, O.Model(cfg, w), prompt, 2, 1e-2, row_tol=2e-2)
    g = gpu_decoder(cfg, w, 1, 0, 2, 0, 640, flags=flags).generate(prompt, 64)
    la = gpu_decoder(cfg, w, 1, W, N, G, 640, flags=flags).generate(prompt, 64)
    assert np.array_equal(la, g)


def test_13b_width_one_layer_slice():
    """Llama-2-13B widths (d 5120, 40 heads x 128, FFN 13824): the GEMMs'
    N and K are not powers of two and 40 heads is not a multiple of the
    attention's head groups; the 1024-token prompt with W=10 N=5 G=10.  One
    layer: on two layers of these random-init weights the bf16 rounding of
    the activations alone (a CPU model of the kernels' rounding points) gives
    0.985e-2 per step, so the GPU's result sits at the 1e-2 bound itself
    (measured 1.0002e-2); the full-depth replay below covers 13B's 40
    layers with the checks that hold at any size."""
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["13b"].sliced(1)
    full = I.make_weights(I.MODELS["13b"], 0, bf16=True, layers=[0])
    w = {k: (v[:1] if isinstance(v, list) else v) for k, v in full.items()}
    prompt = I.make_prompt("13b")
    W, N, G = I.LOOKAHEAD["13b"]
    dec = gpu_decoder(cfg, w, 1, W, N, G, 1152, flags=LA.LA_DEBUG_LOGITS)
    toks, worst = replay_against_oracle(dec, O.Model(cfg, w), prompt, 2, 1e-2, row_tol=2e-2)
    g = gpu_decoder(cfg, w, 1, 0, 2, 0, 1152).generate(prompt, 48)
    la = gpu_decoder(cfg, w, 1, W, N, G, 1152).generate(prompt, 48)
    assert np.array_equal(la, g)


def test_34b_width_one_layer_slice():
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS["34b"].sliced(1)
    full = I.make_weights(I.MODELS["34b"], 0, bf16=True, layers=[0])
    w = {k: (v[:1] if isinstance(v, list) else v) for k, v in full.items()}
    prompt = I.plant_spans(I.zipf_tokens(256, 4000, 1.2, 11), 16, 6, 12)
    W, N, G = I.LOOKAHEAD["34b"]
    flags = LA.LA_PRESEED_PROMPT
    dec = gpu_decoder(cfg, w, 1, W, N, G, 384, flags=flags | LA.LA_DEBUG_LOGITS)
    toks, worst = replay_against_oracle(dec, O.Model(cfg, w), prompt, 2, 1e-2, preseed=True, row_tol=2e-2)
    g = gpu_decoder(cfg, w, 1, 0, 2, 0, 384).generate(prompt, 48)
    la = gpu_decoder(cfg, w, 1, W, N, G, 384, flags=flags).generate(prompt, 48)
    assert np.array_equal(la, g)


@pytest.mark.parametrize("attn", [0, 32], ids=["mma", "attntc"])
@pytest.mark.parametrize("workload,max_seq", [("7b", 768), ("13b", 1024 + 256), ("34b", 2048 + 256)])
def test_full_depth_controller_replay(workload, max_seq, attn):
    """The full-depth models the benchmark times (7B: 32 layers; 13B: 40
    layers, 1024-token prompt; 34B: 48 layers, 8 KV heads, prompt-seeded
    pool, 2048-token prompt), with either attention kernel (the benchmark
    runs the tcgen05 pair)."""
    import oracle as O
    import lossless_lookahead_decoding_gb300 as LA
    cfg = I.MODELS[workload]
    dw = LA.device_weights(cfg, I.iter_weights(cfg, 0, bf16=False), LA.LA_BF16)
    prompt = I.make_prompt(workload)
    W, N, G = I.LOOKAHEAD[workload]
    preseed = workload == "34b"
    flags = (LA.LA_PRESEED_PROMPT if preseed else 0) | attn
    dec = LA.Decoder(cfg, dw, LA.LA_BF16, W, N, G, max_seq, flags=flags)
    ctrl = O.Controller(W, N, G, cfg.vocab)
    ctrl.init(prompt, seed=2, preseed=preseed)
    dec.prefill(prompt)
    assert np.array_equal(dec.window(), ctrl.window())
    c, P = int(prompt[-1]), len(prompt) - 1
    out = []
    for _ in range(24):
        emit = dec.step()
        tok_g, pos_g, ncand = dec.rows()
        amax = dec.argmax()
        tok, pos, _ = ctrl.rows(c, P)
        T = len(tok)
        assert T == 1 + (W + ncand) * (N - 1)
        assert np.array_equal(tok_g[:T], tok) and np.array_equal(pos_g[:T], pos)
        emit_o, _, _ = ctrl.advance(amax[:T])
        assert np.array_equal(emit, emit_o), (emit, emit_o)
        assert np.array_equal(dec.window(), ctrl.window())
        for key in set(int(x) for x in tok):
            assert np.array_equal(dec.pool(key), ctrl.pool(key)), key
        out.extend(emit.tolist())
        P += len(emit)
        c = int(emit[-1])
    dec.close()
    greedy = LA.Decoder(cfg, dw, LA.LA_BF16, 0, 2, 0, max_seq, flags=attn)
    g = greedy.generate(prompt, len(out))
    greedy.close()
    assert np.array_equal(np.array(out, np.int32), g)


def test_7b_width_controller_under_argmax_override():
    """The 121-row step's controller (15 window columns, 15 candidates of 4
    tokens) driven through every acceptance length by overriding the argmaxes,
    against the oracle controller fed the same ones (2-layer 7B slice)."""
    import test_gpu_decode as D
    cfg = I.MODELS["7b"].sliced(2)
    full = I.make_weights(I.MODELS["7b"], 0, bf16=True, layers=[0, 1])
    w = {k: (v[:2] if isinstance(v, list) else v) for k, v in full.items()}
    seen = D._override_replay(cfg, w, 15, 5, 15, 40, seed=8, max_seq=768, prompt=I.make_prompt("7b"))
    assert seen == {1, 2, 3, 4, 5}, seen
