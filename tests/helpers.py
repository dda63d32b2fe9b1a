"""Shared test helpers: build the library, make device models, and replay a GPU
decode against the oracle (controller fed the GPU's argmaxes + step forward)."""
from __future__ import annotations

import numpy as np

import la_inputs as I


def build_lib():
    from lossless_lookahead_decoding_gb300 import build as B
    return B.build()


def gpu_decoder(cfg, weights_np, dtype, W, N, G, max_seq, flags=0, seed=2):
    import lossless_lookahead_decoding_gb300 as LA
    dw = LA.device_weights(cfg, weights_np, dtype)
    return LA.Decoder(cfg, dw, dtype, W, N, G, max_seq, seed=seed, flags=flags)


def rel_l2_rows(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b, axis=-1) / np.maximum(np.linalg.norm(b, axis=-1), 1e-30)


def replay_against_oracle(dec, om, prompt, n_steps, tol, seed=2, preseed=False, check_logits=True, row_tol=None):
    """Run n_steps GPU lookahead steps; after each, check against the oracle:
    rows (tokens/positions), the step's logits (relative L2 error of the
    step's T x V logits <= tol, every step; and every row <= row_tol,
    default tol), emitted tokens and the window/pool state of the oracle
    controller fed the GPU's argmaxes.  Returns (emitted tokens, max step
    logits error)."""
    row_tol = tol if row_tol is None else row_tol
    import oracle as O
    import lossless_lookahead_decoding_gb300 as LA
    W, N, G, V = dec.W, dec.N, dec.G, dec.cfg.vocab
    ctrl = O.Controller(W, N, G, V, variant=O.DIAGONAL if dec.flags & LA.LA_MASK_DIAG else 0)
    ctrl.init(prompt, seed=seed, preseed=preseed)
    seq = O.Seq(om, len(prompt) + n_steps * N + W + N + 8)
    seq.prefill(prompt[:-1])
    dec.prefill(prompt)
    assert np.array_equal(dec.window(), ctrl.window())
    c, P = int(prompt[-1]), len(prompt) - 1
    out, worst = [], 0.0
    for _ in range(n_steps):
        emit_gpu = dec.step()
        tok_g, pos_g, ncand = dec.rows()
        amax_g = dec.argmax()
        tok, pos, vis = ctrl.rows(c, P)
        T = len(tok)
        assert ncand == (T - 1 - W * (N - 1)) // (N - 1)
        assert np.array_equal(tok_g[:T], tok) and np.array_equal(pos_g[:T], pos)
        if check_logits:
            lg_o, _ = seq.step(P, tok, pos, vis)
            lg_g = dec.logits()[:T]
            err = float(np.linalg.norm(lg_g.astype(np.float64) - lg_o) / np.linalg.norm(lg_o.astype(np.float64)))
            worst = max(worst, err)
            assert err <= tol, (err, tol)
            row_err = rel_l2_rows(lg_g, lg_o).max()
            assert row_err <= row_tol, (row_err, row_tol)
        else:
            seq.step(P, tok, pos, vis, want_logits=False)
        emit_o, rows_o, _ = ctrl.advance(amax_g[:T])
        assert np.array_equal(emit_gpu, emit_o), (emit_gpu, emit_o)
        seq.commit(P, rows_o)
        assert np.array_equal(dec.window(), ctrl.window())
        for key in set(int(x) for x in tok):
            assert np.array_equal(dec.pool(key), ctrl.pool(key)), key
        out.extend(emit_gpu.tolist())
        P += len(emit_gpu)
        c = int(emit_gpu[-1])
    return np.array(out, np.int32), worst
